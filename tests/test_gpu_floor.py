"""The decode-floor copy (libropekv_floor.so) that the benchmark times beside
the decode calls copies its bytes exactly, with and without the residency
cap, in the launch shape the benchmark uses (256 CTAs of 192 threads)."""
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from rope_kv_cache_gb300 import build
    build.build_library()


@pytest.mark.parametrize("ctas,threads,cap", [(256, 192, True), (256, 192, False), (7, 32, True),
                                              (1000, 256, True)])
def test_floor_copy_is_a_copy(ctas, threads, cap):
    import rope_kv_cache_gb300 as rk
    n = ctas * threads * 4 * 8                      # int16 elements: 16 B x 4 per thread
    src = torch.randint(-2 ** 15, 2 ** 15, (n,), dtype=torch.int16, device="cuda:0")
    dst = torch.full((n,), 7, dtype=torch.int16, device="cuda:0")
    for _ in range(2):
        rk._binding.ropekv_floor_copy(src, dst, threads, cap)
    torch.cuda.synchronize()
    assert torch.equal(src, dst)
