// Profiling hooks, compiled in only when SGB_TRACE_ENABLED is defined: per-CTA
// phase timestamps and cycle counters written to a 32-slot row per CTA of the
// kernel parameter block's `trace` buffer.  Release builds expand every macro
// to nothing.
#pragma once

#include "ptx.cuh"

// Phase timestamps for profiling builds (compiled with SGB_TRACE_ENABLED):
// slot `slot` of CTA blockIdx.x gets the global timer when `cond` holds.
#ifdef SGB_TRACE_ENABLED
#define SGB_TRACE(kp, cond, slot)                                                               \
    do {                                                                                        \
        if ((kp).trace && (cond)) (kp).trace[static_cast<size_t>(blockIdx.x) * 32 + (slot)] =   \
            ::sgb::ptx::globaltimer();                                                          \
    } while (0)
// Cycle accounting for profiling builds: SGB_CYCLES_BEGIN(t) starts a stopwatch,
// SGB_CYCLES_END(acc, t) adds the elapsed SM cycles to a local accumulator that
// SGB_TRACE_VALUE stores in the trace slot at the end.
#define SGB_CYCLES_BEGIN(t) const uint64_t t = ::sgb::ptx::clock64()
#define SGB_CYCLES_END(acc, t) (acc) += ::sgb::ptx::clock64() - (t)
#define SGB_TRACE_VALUE(kp, cond, slot, value)                                                   \
    do {                                                                                        \
        if ((kp).trace && (cond)) (kp).trace[static_cast<size_t>(blockIdx.x) * 32 + (slot)] = (value); \
    } while (0)
// Per-stage timeline of CTA 0 (stages < 256): role r of stage i at
// trace[8192 + 4*i + r] (0 activation issue, 1 weight issue, 2 data landed
// (waiter), 3 MMA start).
#define SGB_STAGE_MARK(kp, i, r)                                                                \
    do {                                                                                        \
        if ((kp).trace && blockIdx.x == 0 && (i) < 256)                                        \
            (kp).trace[8192 + 4 * static_cast<size_t>(i) + (r)] = ::sgb::ptx::globaltimer();    \
    } while (0)
// Per-stage timeline of CTA pair 0 (stages < 256): event r (< 8) of stage i at
// trace[8192 + 8*i + r].
#define SGB_PAIR_MARK(kp, i, r)                                                                 \
    do {                                                                                        \
        if ((kp).trace && blockIdx.x < 2 && (i) < 256)                                          \
            (kp).trace[8192 + 8 * static_cast<size_t>(i) + (r)] = ::sgb::ptx::globaltimer();    \
    } while (0)
#else
#define SGB_PAIR_MARK(kp, i, r) \
    do {                        \
    } while (0)
#define SGB_STAGE_MARK(kp, i, r) \
    do {                         \
    } while (0)
#define SGB_TRACE(kp, cond, slot) \
    do {                          \
    } while (0)
#define SGB_CYCLES_BEGIN(t) \
    do {                    \
    } while (0)
#define SGB_CYCLES_END(acc, t) \
    do {                       \
    } while (0)
#define SGB_TRACE_VALUE(kp, cond, slot, value) \
    do {                                       \
    } while (0)
#endif
