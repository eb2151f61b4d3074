/*
 * ropekv_floor.h -- C ABI of libropekv_floor.so, a measurement reference for
 * the decode-sized launches of libropekv.so. It is not part of the fused
 * RoPE + KV-cache write (the pages have no counterpart): it is the floor that
 * one such launch cannot go below.
 *
 * ropekv_floor_copy copies `bytes` bytes from src to dst with the launch shape
 * and launch policy of libropekv's decode-sized launches: CTAs of
 * `threadsPerCta` threads, four 16-byte vectors per thread (a decode thread
 * loads and stores two items of two vectors), an L2 prefetch of the thread's
 * source vectors before the dependent-launch wait, the programmatic
 * dependent-launch attribute, L1-bypassing evict-first loads and evict-first
 * stores, and (when `cap` is non-zero) the same residency cap: dynamic shared
 * memory that the kernel does not use, sized so that at most
 * ceil(grid / SMs) CTAs fit on one SM. What it leaves out is exactly the
 * decode kernel's own work: the position chain, the cos/sin loads and the
 * rotation. So a chain of these copies, timed like the decode calls, gives the
 * shortest time a dependent launch moving the same bytes in the same grid
 * takes on the device.
 *
 *   src, dst       device pointers, 16-byte aligned, not overlapping; owned by
 *                  the caller.
 *   bytes          a positive multiple of 16 * 4 * threadsPerCta (whole CTAs).
 *   threadsPerCta  a multiple of 32 in [32, 256].
 *   cap            non-zero: reserve the residency cap's shared memory.
 *   stream         a cudaStream_t passed as void* (NULL = legacy default).
 * Returns 0, -1 (NULL pointer), -2 (misaligned), -6 (bad size) or -10 (the
 * launch failed, read from the launch's own result). Allocates nothing,
 * never synchronises; the current device must hold the buffers.
 */
#ifndef ROPEKV_FLOOR_H
#define ROPEKV_FLOOR_H

#include <stdint.h>

#if defined(__GNUC__)
#define ROPEKV_FLOOR_API __attribute__((visibility("default")))
#else
#define ROPEKV_FLOOR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

ROPEKV_FLOOR_API int ropekv_floor_copy(const void* src, void* dst, int64_t bytes,
                                       int32_t threadsPerCta, int32_t cap, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ROPEKV_FLOOR_H */
