/*
 * specverify_internal.h -- tuning and test hooks of libspecverify.so. Not part of the C ABI in
 * include/specverify.h: production callers need neither; the tests and the tuning scripts use them to pin
 * a launch shape and to read back the launch plan. Both act on state shared by every thread of the process.
 */
#ifndef SPECVERIFY_INTERNAL_H
#define SPECVERIFY_INTERNAL_H

#ifdef __cplusplus
extern "C" {
#endif

/* Forces the number of CTAs of the statistics pass of spec_verify, spec_cactus_verify, spec_cactus_kl_verify,
 * spec_verify_filtered and spec_verify_static (1 to 1024; 0 restores the automatic choice, every SM once). The
 * grid fixes how the rows are cut into per-warp segments, so results depend on it only through
 * floating-point summation order. Process-wide and not synchronised: set it while no other thread calls the
 * library. Returns 0, or -1 for an unsupported value. */
int spec_debug_set_stats_grid(int ctas);

/* The launch plan of the last call made on this thread, as five ints: 0, ring slots per warp, CTAs
 * launched, kernel (0: the statistics pass of spec_verify / spec_cactus_verify / spec_verify_static; 2: the
 * gamma kernel of spec_counterfactual_gamma, which parks rows in tensor memory; 3: the argmax pass of
 * spec_greedy_verify; 5: the one-launch gamma and chain kernel; 6: spec_verify_filtered through the
 * line-maxima bound kernel, then the radix threshold kernel on the rows it left; 7: spec_verify_filtered
 * through the radix threshold kernel alone), pieces per row. out5 is host memory.
 * Returns 0, or -1 for a NULL pointer. */
int spec_debug_last_plan(int* out5);

/* Sets the chunk mass (sum of the target and draft probabilities of an 8-logit chunk) above which the residual
 * draw evaluates the chunk in float-float instead of float (0 restores the default). Larger values are faster
 * and leave more elements to the float path. Process-wide and not synchronised. Returns 0, or -1 for a
 * negative or NaN value. */
int spec_debug_set_draw_tau(float tau);

/* 1: spec_counterfactual_gamma with a selected drafter (rows aligned for bulk copies) runs the gamma pass
 * and the selected drafter's chain and draw as one cooperative launch (a grid barrier between the two, one
 * CTA per sequence for the draw, the barrier's words in the workspace header, which spec_clear_status
 * zeroes); 0 (the default): the gamma kernel, then the draw kernel with programmatic dependent launch.
 * Process-wide and not synchronised. Returns 0, or -1 for another value. */
int spec_debug_set_gamma_one_launch(int on);

/* The residual draw's float-float building block on n inputs (device pointers): out[2i], out[2i + 1] = the
 * float pair of 2^((d[i]) c + l) with c = log2(e) / temperature and l = l_hi[i] + l_lo[i], evaluated as the
 * draw evaluates its large elements. Asynchronous on `stream`. Returns 0, or -1 for bad arguments or a launch
 * failure. */
int spec_debug_exp2ff(const float* d, const float* l_hi, const float* l_lo, float* out, int n, float temperature,
                      void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_INTERNAL_H */
