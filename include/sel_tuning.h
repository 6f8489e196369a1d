/*
 * sel_tuning.h -- tuning and test hooks of libsel.  Normal callers need none
 * of this: without it every call takes the automatic launch plan.
 *
 * The pages have no counterpart: the tutorial's library picks its kernels
 * itself.  These knobs exist so that tests can run every kernel on the same
 * shapes, and so that measurements can compare plans.
 *
 * The knobs start from the environment, read once when the library first
 * plans a call: SEL_PLAN=reg|row|wide|split|stream|flat, SEL_PARTS=n,
 * SEL_ROW_SAMPLE=1, SEL_HIST_AGG=1, SEL_ROW_ORDER=1.  sel_set_tuning changes them at any time
 * after that; plans are cached per knob setting, so a change takes effect on
 * the next call.  They are process-wide (not per thread).
 */
#ifndef SEL_TUNING_H_
#define SEL_TUNING_H_

#include "sel.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Knobs. */
enum {
    SEL_TUNE_PLAN = 0,       /* a SEL_PLAN_* value: force one kernel where it can run the shape */
    SEL_TUNE_PARTS = 1,      /* > 0: parts per row of the streaming kernel's split mode; 0 = automatic */
    SEL_TUNE_ROW_SAMPLE = 2, /* 1: the staged row kernel estimates its first digit from a sample */
    SEL_TUNE_HIST_AGG = 3,   /* 1: first-pass histograms with warp-aggregated atomics */
    SEL_TUNE_ROW_ORDER = 4   /* 1: with per-row ends, CTAs take rows from both ends of the batch
                                alternately; 0 (default): in order -- measured faster on causal
                                row ends, where neighbouring rows share memory traffic */
};

/* Values of SEL_TUNE_PLAN.  A forced kernel that cannot run a shape leaves
 * that shape to the automatic plan. */
enum {
    SEL_PLAN_AUTO = -1,
    SEL_PLAN_REG = 0,    /* one CTA per row, row held in registers (rows of at most 16 KB) */
    SEL_PLAN_ROW = 1,    /* one CTA per row, row staged in shared memory */
    SEL_PLAN_WIDE = 2,   /* one streaming pass per row (or per part of a row) */
    SEL_PLAN_SPLIT = 3,  /* staged slices of a row over several CTAs */
    SEL_PLAN_STREAM = 4, /* exact passes over global memory */
    SEL_PLAN_FLAT = 5    /* rows cut into chunks dealt over one resident CTA per SM */
};

/* Sets a knob.  SEL_OK, or SEL_EINVAL for an unknown knob or value. */
SEL_API int sel_set_tuning(int knob, int value);

/* A knob's current value, or -1 for an unknown knob. */
SEL_API int sel_get_tuning(int knob);

/* 1 when this library is the debug build (libsel_debug.so, compiled with
 * SEL_DEBUG): its kernels check their staged-list and region offsets,
 * workspace slots, output positions and gathered key rows before each
 * access, skip an access that would fall outside its buffer and write
 * SEL_EBOUNDS to err_flag.  0 for the normal build, where those checks are
 * compiled away. */
SEL_API int sel_debug_build(void);

/* Test of the failure path of the kernels' bounded waits (the tutorial's
 * kernel traps on a NaN; this library never traps, and every wait on a
 * barrier gives up after a bound and reports SEL_ETIMEOUT instead).  Launches
 * on `stream` one CTA that waits, with a budget of `cycles` GPU clock cycles,
 * on a barrier armed for 16 bytes that no copy ever delivers (none is issued,
 * so nothing lands after the wait gives up).  The wait runs out, writes
 * SEL_ETIMEOUT to the caller-owned, zeroed *err_flag and the CTA returns;
 * the stream and the context stay usable.  Returns SEL_EINVAL for a NULL
 * err_flag or negative cycles, SEL_ECUDA if the launch fails, else SEL_OK
 * (asynchronous: read err_flag after synchronising). */
SEL_API int sel_selftest_wait_timeout(int32_t *err_flag, long long cycles, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SEL_TUNING_H_ */
