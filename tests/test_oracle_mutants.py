"""The oracle's pins catch planted mistakes.

Each case copies the oracle's C source, plants one plausible mistake (a
dropped term, a wrong sign or partner, a wrong index, a slot off by one, ...),
builds it into a temporary library and runs the oracle pin tests against that
build in a child process. Every mutant must make at least one pin fail. The
real oracle is never modified; everything here runs on the CPU.
"""
import os
import shutil
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ropekv_oracle.c")
HDR = os.path.join(ROOT, "oracle", "ropekv_oracle.h")
PIN_TESTS = ["tests/test_oracle_rope.py", "tests/test_oracle_entries.py",
             "tests/test_oracle_dflash.py", "tests/test_oracle_slotmap.py",
             "tests/test_oracle_qknorm.py", "tests/test_oracle_fp8.py",
             "tests/test_oracle_fp16.py", "tests/test_oracle_cross_entry.py"]

MUTANTS = {
    "neox_rotate_sign": ("out[d] = (d < h) ? -x[d + h] : x[d - h];",
                         "out[d] = (d < h) ? x[d + h] : x[d - h];"),
    "gptj_rotate_partner": ("out[d] = (d % 2 == 0) ? -x[d + 1] : x[d - 1];",
                            "out[d] = (d % 2 == 0) ? -x[d + 1] : -x[d - 1];"),
    "neox_freq_index": ("return (style == STYLE_NEOX) ? (d % h) : (d / 2);",
                        "return (style == STYLE_NEOX) ? (d / 2) : (d / 2);"),
    "gptj_freq_index": ("return (style == STYLE_NEOX) ? (d % h) : (d / 2);",
                        "return (style == STYLE_NEOX) ? (d % h) : (d % h);"),
    "cos_sin_swapped": ("double c = (double)cs_row[f];\n        double s = (double)cs_row[h + f];",
                        "double c = (double)cs_row[h + f];\n        double s = (double)cs_row[f];"),
    "dropped_sin_term": ("y[d] = x[d] * c + rot[d] * s;", "y[d] = x[d] * c;"),
    "rounding_truncates": ("double q = nearbyint(ldexp(a, 10 - E));",
                           "double q = floor(ldexp(a, 10 - E));"),
    "subnormal_scale": ("double k = nearbyint(ldexp(a, 24));",
                        "double k = nearbyint(ldexp(a, 23));"),
    "continuous_slot_off_by_one": (
        "long long slot = (long long)kvCacheEndLens[b] - S + s;\n            long long pos = slot;",
        "long long slot = (long long)kvCacheEndLens[b] - S + s + 1;\n            long long pos = slot;"),
    "tree_position_from_slot": ("long long pos = tokenPosIds[(size_t)b * S + s];",
                                "long long pos = (long long)kvCacheEndLens[b] - S + s;"),
    "v_from_k_head": ("qkv_tok + (size_t)(Hq + Hkv + hv) * D",
                      "qkv_tok + (size_t)(Hq + hv) * D"),
    "packed_k_not_in_place": ("if (k_in_place)", "if (0)"),
    "paged_row_by_position": ("tokenAlignedCosSin + (size_t)t * r;",
                              "tokenAlignedCosSin + (size_t)(pos % numDeltaTokens) * r;"),
    "paged_v_plane_unchecked": ("if (idV >= numPages && (int64_t)idV < 2 * (int64_t)numPages)",
                                "if (idV >= 0 && (int64_t)idV < 2 * (int64_t)numPages)"),
    "paged_capacity_unchecked": ("if (lp >= maxPagesPerSeq)", "if (lp > maxPagesPerSeq)"),
    "capacity_rule_inclusive": ("return cosSinSeqLen > kvCapacity ? 1 : 0;",
                                "return cosSinSeqLen >= kvCapacity ? 1 : 0;"),
    "metadata_position_base": ("deltaPositions[t] = oldDraftCacheLengths[b] + j;",
                               "deltaPositions[t] = oldDraftCacheLengths[b] + j + 1;"),
    "metadata_length_off_by_one": ("if (j < len) {", "if (j <= len) {"),
    "gather_state_ignored": ("state = stateIndices[seq];", "state = seq;"),
    "gather_capacity_unchecked": ("seq < batchSize && pos < cacheCapacity;",
                                  "seq < batchSize && pos <= cacheCapacity;"),
    "gather_shared_row_ignored": ("state = (sourceRows == 1) ? 0 : seq;", "state = seq;"),
    "slotmap_block_offset_swapped": ("int64_t block = slot / blockSize;\n        int64_t off = slot % blockSize;",
                                     "int64_t block = slot % blockSize;\n        int64_t off = slot / blockSize;"),
    "slotmap_negative_slot_written": ("if (slot < 0 || slot >= slots)", "if (slot >= slots)"),
    "rmsnorm_mean_not_divided": ("double inv = 1.0 / sqrt(ss / D + eps);",
                                 "double inv = 1.0 / sqrt(ss + eps);"),
    "rmsnorm_eps_dropped": ("double inv = 1.0 / sqrt(ss / D + eps);",
                            "double inv = 1.0 / sqrt(ss / D);"),
    "qknorm_weights_swapped": ("norm_rope_head_f16(tok + (size_t)hq * D, qNormWeight,",
                               "norm_rope_head_f16(tok + (size_t)hq * D, kNormWeight,"),
    "e4m3_no_saturation": ("if (field > 15 || (field == 15 && q - 8.0 > 6.0))", "if (field > 16)"),
    "e4m3_truncates": ("double q = nearbyint(ldexp(a, 3 - E));", "double q = floor(ldexp(a, 3 - E));"),
    "e4m3_subnormal_scale": ("double k = nearbyint(ldexp(a, 9));", "double k = nearbyint(ldexp(a, 8));"),
    "fp8_scale_not_inverted": ("kc[d] = ropekv_oracle_f64_to_e4m3(y[d] * (1.0 / (double)kScale));",
                               "kc[d] = ropekv_oracle_f64_to_e4m3(y[d] * (double)kScale);"),
    "slotmap_stride_ignored": ("rope_head_f16(k + (size_t)t * kStride", "rope_head_f16(k + (size_t)t * Hkv * D"),
    "cs_batch_ignored": ("int bc = (csBatch == 1) ? 0 : b;", "int bc = 0;"),
    "qknorm_tail_copied": ("for (int d = 0; d < D; ++d)\n        dst[d] = ropekv_oracle_f64_to_f16(y[d]);",
                           "for (int d = 0; d < D; ++d)\n        dst[d] = (d < r) ? ropekv_oracle_f64_to_f16(y[d]) : src[d];"),
    "qknorm_after_rotation": ("ropekv_oracle_rms_norm_f64(x, weight, eps, D, n);\n    ropekv_oracle_rope_head_f64(n, cs, D, r, style, y);",
                              "ropekv_oracle_rope_head_f64(x, cs, D, r, style, n);\n    ropekv_oracle_rms_norm_f64(n, weight, eps, D, y);"),
    "qknorm_pos_upper_unchecked": ("long long slot = pos;\n            if (slot < 0 || slot >= cap || pos >= csSeq)",
                                   "long long slot = pos;\n            if (slot < 0 || slot >= cap)"),
    "tree_pos_upper_unchecked": ("if (pos < 0 || pos >= csSeq || slot < 0 || slot >= cap)",
                                 "if (pos < 0 || slot < 0 || slot >= cap)"),
    "fp8_pos_upper_unchecked": ("if (slot < 0 || slot >= cap || slot >= csSeq)",
                                "if (slot < 0 || slot >= cap)"),
    "dims_cs_batch_unchecked": ("if (csBatch != 1 && csBatch != B)\n        return 0;", ""),
    "dims_gqa_ratio_unchecked": ("if (Hq % Hkv != 0)\n        return 0;", ""),
    "dims_odd_rotary_accepted": ("if (r <= 0 || r % 2 != 0 || r > D)\n        return 0;\n    if (csBatch",
                                 "if (r <= 0 || r > D)\n        return 0;\n    if (csBatch"),
    "f16_nan_signaling": ("return (uint16_t)(sign | 0x7E00u);", "return (uint16_t)(sign | 0x7C01u);"),
    "fp8_k_rounded_through_f16": (
        "kc[d] = ropekv_oracle_f64_to_e4m3(y[d] * (1.0 / (double)kScale));",
        "kc[d] = ropekv_oracle_f64_to_e4m3(ropekv_oracle_f16_to_f64(ropekv_oracle_f64_to_f16(y[d])) * (1.0 / (double)kScale));"),
    "fp8_v_uses_k_scale": ("(1.0 / (double)vScale));", "(1.0 / (double)kScale));"),
    "gather_seq_upper_unchecked": ("int ok = pos >= 0 && seq >= 0 && seq < batchSize && pos < cacheCapacity;",
                                   "int ok = pos >= 0 && seq >= 0 && pos < cacheCapacity;"),
    "gather_invalid_row_not_zero": ("+ pos) * rotaryDim + d] : 0.0f;", "+ pos) * rotaryDim + d] : 1.0f;"),
    "paged_k_plane_inclusive": ("if (idK >= 0 && idK < numPages) {", "if (idK >= 0 && idK <= numPages) {"),
    "paged_v_plane_low_exclusive": ("if (idV >= numPages && (int64_t)idV < 2 * (int64_t)numPages)",
                                    "if (idV > numPages && (int64_t)idV < 2 * (int64_t)numPages)"),
    "paged_table_plane_major": (
        "int32_t idK = pageTable[((size_t)seq * 2 + 0) * maxPagesPerSeq + lp];\n        int32_t idV = pageTable[((size_t)seq * 2 + 1) * maxPagesPerSeq + lp];",
        "int32_t idK = pageTable[((size_t)0 * batchSize + seq) * maxPagesPerSeq + lp];\n        int32_t idV = pageTable[((size_t)1 * batchSize + seq) * maxPagesPerSeq + lp];"),
    "metadata_sequence_is_row": ("deltaTokenToSequence[t] = b;", "deltaTokenToSequence[t] = j;"),
    "rmsnorm_eps_not_passed": ("ropekv_oracle_rms_norm_f64(x, weight, eps, D, n);",
                               "ropekv_oracle_rms_norm_f64(x, weight, 1e-6, D, n);"),
    "slotmap_v_stride_ignored": ("memcpy(vc, v + (size_t)t * vStride", "memcpy(vc, v + (size_t)t * kStride"),
    "slotmap_q_skipped_with_cache": (
        "        const float* cs = cosSin + (size_t)pos * r;\n        for (int hq = 0; hq < Hq; ++hq)",
        "        const float* cs = cosSin + (size_t)pos * r;\n        if (slotMapping[t] < 0)\n            continue;\n        for (int hq = 0; hq < Hq; ++hq)"),
    "cache_plane_head_swapped": ("return ((((size_t)b * 2 + plane) * Hkv + hk) * (size_t)cap + slot) * (size_t)D;",
                                 "return ((((size_t)b * Hkv + hk) * 2 + plane) * (size_t)cap + slot) * (size_t)D;"),
    "tree_slot_from_position": ("long long slot = (long long)kvCacheEndLens[b] - S + s;\n            if (pos < 0",
                                "long long slot = pos;\n            if (pos < 0"),
    "fp8_tail_not_scaled": ("kc[d] = ropekv_oracle_f64_to_e4m3(y[d] * (1.0 / (double)kScale));",
                            "kc[d] = ropekv_oracle_f64_to_e4m3(d < r ? y[d] * (1.0 / (double)kScale) : y[d]);"),
    "packed_table_length_unchecked": ("if (S > cap || S > csSeq)", "if (S > cap)"),
    "gather_source_transposed": ("source[((size_t)state * cacheCapacity + pos) * rotaryDim + d]",
                                 "source[((size_t)pos * sourceRows + state) * rotaryDim + d]"),
    "slotmap_cache_head_major": (
        "uint16_t* kc = keyCache + (((size_t)block * blockSize + off) * Hkv + hk) * D;",
        "uint16_t* kc = keyCache + (((size_t)block * Hkv + hk) * blockSize + off) * D;"),
    "qknorm_norm_over_rotary_only": (
        "ropekv_oracle_rms_norm_f64(x, weight, eps, D, n);",
        "ropekv_oracle_rms_norm_f64(x, weight, eps, r, n);\n    for (int d = r; d < D; ++d)\n        n[d] = x[d] * ropekv_oracle_f16_to_f64(weight[d]);"),
    "sin_index_mirrored": ("double s = (double)cs_row[h + f];", "double s = (double)cs_row[r - 1 - f];"),
}


def _run_mutant(name, workdir):
    """Build one mutant into its own library and run the pins against it in a
    child process; returns (returncode, stdout)."""
    old, new = MUTANTS[name]
    src = open(SRC).read()
    if src.count(old) != 1:
        return None, f"mutation site for {name} found {src.count(old)} times"
    mdir = os.path.join(workdir, name)
    os.makedirs(mdir, exist_ok=True)
    shutil.copy(HDR, mdir)
    msrc = os.path.join(mdir, "ropekv_oracle.c")
    with open(msrc, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(mdir, "libmutant.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", lib, msrc, "-lm"], check=True)
    env = dict(os.environ, ROPEKV_ORACLE_LIB=lib)
    proc = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                           *PIN_TESTS], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=900)
    return proc.returncode, proc.stdout + proc.stderr


@pytest.fixture(scope="module")
def results():
    """Every mutant's pin run, side by side (each is an independent child
    process on its own copy of the oracle)."""
    d = tempfile.mkdtemp(prefix="ropekv_mutants_")
    try:
        workers = max(1, min(8, os.cpu_count() or 1))
        with ThreadPoolExecutor(workers) as ex:
            futs = {n: ex.submit(_run_mutant, n, d) for n in MUTANTS}
            yield {n: f.result() for n, f in futs.items()}
    finally:
        shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, results):
    rc, out = results[name]
    assert rc is not None, out
    assert rc != 0, f"mutant {name} passed every pin:\n{out[-2000:]}"
    # a mistake that writes outside its buffer may kill the child by a signal
    # before pytest reports; that is caught as well
    killed = rc < 0 or rc >= 128
    assert killed or "failed" in out or "error" in out.lower(), out[-2000:]
