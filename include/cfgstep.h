/*
 * cfgstep.h -- C ABI of the classifier-free-guidance (CFG) sampler step for
 * one NVIDIA B300 (sm_103a).
 *
 * One denoising step of a CFG diffusion sampler, run once per step over the
 * whole latent, as every multi-GPU scheme on the source pages runs it after
 * the conditional and unconditional predictions are gathered (xDiT review,
 * section 3 "CFG Parallelism": the gather happens before the scheduler):
 *
 *   1. rel-MAE, the denoising discrepancy between the two predictions
 *      (Hybridiff notes, "Accelerating Diffusion via Hybrid Data-Pipeline
 *      Parallelism Based on Conditional Guidance Scheduling", key design 2):
 *        M_s = sum|p_c - p_u| / sum|p_u|   over the whole latent;
 *   2. the tau1/tau2 schedule (same notes, key design 3), kept on the device:
 *        G_s = (M_s - M_{s-L}) / L, tau1' = first s with 0 <= G_s < g_slope,
 *        tau1 = min(tau1', tau_cap), tau2 = tau1 + k;
 *   3. guidance  e = p_u + w (p_c - p_u);
 *   4. the update: DDIM with eta >= 0 (zyxy.net "AIGC text-to-image: how to
 *      speed up diffusion-model inference", section 3, DDIM sampler), or an
 *      Euler step of a flow-matching ODE with the velocity pair (Hybridiff
 *      notes, "Loss / training strategy").
 *
 * Conventions for every entry point below:
 *   - Tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or keeps them.  Parameter structs
 *     (cfg_sched_params) and tables marked "host" are read on the host
 *     during the call and not kept.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All device work is enqueued asynchronously on it; no call
 *     synchronises the host except where stated.
 *   - Latents are dense, contiguous arrays of `n` elements in any order the
 *     caller likes (the step is elementwise apart from the global sums), in
 *     fp32 (CFG_F32) or bf16 (CFG_BF16).  Arithmetic is fp32; the rel-MAE
 *     sums are carried in double-fp32 (about 48 significant bits) and their
 *     ratio M is returned as an fp64 value within about 2^-44 of the
 *     quotient of the two sums; the slope G = (M_s - M_{s-L}) / L is the
 *     IEEE fp64 result (each operation correctly rounded).  Sums must stay
 *     within the fp32 range.  16-byte aligned pointers take the 128-bit
 *     vector path; any other alignment is accepted and takes a scalar path.
 *   - `x_out` may alias `x_in` (in-place update).
 *   - Return value: CFG_OK (0) or a negative cfg_status.  On error nothing
 *     has been enqueued, and cfg_last_error() (per host thread) describes
 *     the failure.  CFG_ERR_CUDA reports an error returned by the CUDA
 *     runtime while enqueuing (asynchronous kernel faults surface at the
 *     caller's next synchronisation, as usual in CUDA).
 */
#ifndef CFGSTEP_H
#define CFGSTEP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define CFG_API __attribute__((visibility("default")))
#else
#define CFG_API
#endif

/* Storage types.  CFG_BF16 and CFG_BF16_EXACT store the same bf16 values in
 * memory and differ only in how a step rounds its result (see
 * cfg_ddim_step): CFG_BF16 rounds the fp32 evaluation of the step once
 * (within one bf16 ulp of the exact step); CFG_BF16_EXACT rounds the exact
 * step correctly (as an fp64 evaluation rounded once to bf16), at some cost
 * in time.  Reductions treat the two alike. */
enum cfg_dtype { CFG_F32 = 0, CFG_BF16 = 1, CFG_BF16_EXACT = 2 };

/* Sampler kinds for cfg_sampler_run. */
enum cfg_mode { CFG_MODE_DDIM = 0, CFG_MODE_FLOW = 1 };

/* Status codes. */
enum cfg_status {
  CFG_OK = 0,
  CFG_ERR_INVALID_ARG = -1,       /* a pointer, size or parameter is out of range */
  CFG_ERR_UNSUPPORTED_DTYPE = -2, /* dtype is not one of cfg_dtype */
  CFG_ERR_WORKSPACE = -3,         /* workspace missing, too small or misaligned */
  CFG_ERR_CUDA = -4,              /* the CUDA runtime returned an error */
  CFG_ERR_CALLBACK = -5           /* the denoiser callback returned non-zero */
};

/* "Undefined / never" value of the tau fields. */
#define CFG_TAU_NONE 2147483647

/* Longest run the device-side schedule records. */
#define CFG_SCHED_MAX_STEPS 1024

/* Phase of a step (Hybridiff notes, "Overall framework"):
 * Warm-Up [T, tau1], Parallelism (tau1, tau2), Fully-Connecting [tau2, 0],
 * in step indices: s <= tau1, tau1 < s < tau2, s >= tau2. */
enum cfg_phase { CFG_PHASE_WARMUP = 0, CFG_PHASE_PARALLEL = 1, CFG_PHASE_FULL = 2 };

/* cfg_sched_state.flags bits. */
#define CFG_SCHED_FLAG_OUT_OF_ORDER 1u /* a step index arrived that was not n_seen */
#define CFG_SCHED_FLAG_DEFER_CLASH 2u  /* a deferred step was followed by a launch on the same
                                          workspace writing the same partial slot (a step of the
                                          same parity); its rel-MAE was dropped */

/* cfg_sched_params.flags bits. */
#define CFG_SCHED_DEFER 1u /* defer each step's rel-MAE to the next launch (see below) */

/*
 * Parameters of the tau1/tau2 rule (Hybridiff notes, key design 3).  Host
 * struct, read during the call.
 *   L        slope window in steps, >= 1;
 *   k        tau2 = tau1 + k, >= 0 (the notes' sweet spot is k = 5);
 *   g_slope  slope threshold, finite;
 *   tau_cap  >= 0: a calibrated safety cap (the step index of the minimum of
 *            a previously measured discrepancy curve); -1: the earliest
 *            argmin of this run's own rel-MAE trace, known after the last step;
 *   n_steps  steps in the run, 1..CFG_SCHED_MAX_STEPS;
 *   flags    0, or CFG_SCHED_DEFER: every step except the run's last leaves
 *            the combine of its rel-MAE partial sums (and the M_out and M[s]
 *            writes of that step) to the next launch on the same workspace,
 *            and that launch leaves the step's schedule update to the launch
 *            after it; each is done in a side block while those launches
 *            stream their own data, so neither the reduction's latency nor
 *            the rule's leaves a mark on the critical path.  The next launch
 *            on that workspace must be the next step (the other step
 *            parity), a call that finishes in-launch (a non-deferred step,
 *            cfg_relmae_reduce), or cfg_workspace_flush; a same-parity
 *            deferred step instead drops it and sets
 *            CFG_SCHED_FLAG_DEFER_CLASH.  A launch that does not defer (the
 *            last step of the run, n_steps - 1, always finishes in-launch)
 *            completes all pending work first, so a finished run's state is
 *            complete;
 *   reserved must be 0.
 * The "t" of the notes' rule is read as the step index s, counted from the
 * first denoising step (s = 0 at the noisiest timestep).
 */
typedef struct cfg_sched_params {
  int32_t L;
  int32_t k;
  double g_slope;
  int32_t tau_cap;
  int32_t n_steps;
  uint32_t flags;
  int32_t reserved;
} cfg_sched_params;

/*
 * Device-resident schedule state, one per sampler run (caller-allocated
 * device memory of sizeof(cfg_sched_state) bytes, 16-byte aligned; contents
 * need no initialisation: step 0 resets it).  Updated by one device thread
 * after each step's rel-MAE is known; the host reads it whenever it likes.
 *   n_seen      steps recorded (the next expected step index);
 *   tau1p       tau1' (CFG_TAU_NONE until found);
 *   argmin      earliest index of the smallest non-NaN M so far (-1: none);
 *   tau_cap     the cap used (CFG_TAU_NONE until decided);
 *   tau1, tau2  CFG_TAU_NONE until decided;
 *   decided_at  step at which tau1/tau2 became final (-1 before): with a
 *               calibrated cap, min(tau1', tau_cap); otherwise the last step;
 *   flags       CFG_SCHED_FLAG_* bits;
 *   min_M       the smallest M so far;
 *   M[s]        rel-MAE trace; G[s] slope (NaN for s < L);
 *   phase[s]    cfg_phase of each step, written at the last step.
 * NaN compares false everywhere (a NaN M never sets tau1' or the argmin).
 */
typedef struct cfg_sched_state {
  int32_t n_seen;
  int32_t tau1p;
  int32_t argmin;
  int32_t tau_cap;
  int32_t tau1;
  int32_t tau2;
  int32_t decided_at;
  uint32_t flags;
  double min_M;
  double M[CFG_SCHED_MAX_STEPS];
  double G[CFG_SCHED_MAX_STEPS];
  uint8_t phase[CFG_SCHED_MAX_STEPS];
  uint8_t pad[8]; /* sizeof is a multiple of 16, so arrays of states stay 16-byte aligned */
} cfg_sched_state;

/*
 * Bytes of device workspace a step or reduction over `n` elements of
 * `dtype` needs (a header with a completion counter and the descriptor of a
 * deferred reduction, then three slots of per-block partial sums).  The value does not depend on the device.  Returns 0
 * for an unsupported dtype or n < 0.
 */
CFG_API size_t cfg_workspace_bytes(int64_t n, int32_t dtype);

/*
 * Prepare a workspace for first use: zero its completion counter on
 * `stream`.  Call once per workspace buffer (a zero-filled buffer is
 * already prepared); every later call leaves the counter at zero again.
 * ws: device, 16-byte aligned, ws_bytes >= cfg_workspace_bytes(...).
 * One workspace must not be used by two calls that may run concurrently.
 */
CFG_API int cfg_workspace_init(void* ws, size_t ws_bytes, void* stream);

/*
 * Complete the work steps launched with CFG_SCHED_DEFER left in the
 * workspace (a pending rel-MAE with its M_out write, and pending schedule
 * updates); a no-op when none is pending.  One single-block launch on
 * `stream`.
 */
CFG_API int cfg_workspace_flush(void* ws, size_t ws_bytes, void* stream);

/*
 * rel-MAE alone (Hybridiff notes, key design 2; with the velocity pair for
 * flow models, "Loss / training strategy"):
 *   M = sum_i |pred_c[i] - pred_u[i]| / sum_i |pred_u[i]|
 * with 0/0 -> 0 and x/0 -> +inf; otherwise IEEE: an infinite prediction
 * makes its sum +inf (so M = +inf, or NaN for inf/inf), and a NaN makes M NaN.
 *   pred_c, pred_u  device, n elements of dtype;
 *   M_out           device double, nullable: receives M;
 *   st, sp          nullable together: when given, M is recorded as step
 *                   `step` of the schedule (0 <= step < sp->n_steps);
 *   ws, ws_bytes    device workspace (cfg_workspace_bytes, cfg_workspace_init).
 * Reads 2n elements; one fused pass plus an in-kernel fixed-order fp64
 * combine of the block partials (deterministic for a given device).
 */
CFG_API int cfg_relmae_reduce(const void* pred_c, const void* pred_u, int64_t n, int32_t dtype,
                              double* M_out, cfg_sched_state* st, const cfg_sched_params* sp,
                              int32_t step, void* ws, size_t ws_bytes, void* stream);

/*
 * One fused CFG + DDIM step (zyxy.net DDIM sampler, section 3):
 *   e      = pred_u + w (pred_c - pred_u)
 *   sigma  = eta sqrt((1 - abar_prev)/(1 - abar_t) (1 - abar_t/abar_prev))
 *   x0     = (x - sqrt(1 - abar_t) e) / sqrt(abar_t)
 *   x_out  = sqrt(abar_prev) x0 + sqrt(1 - abar_prev - sigma^2) e + sigma z
 * abar_prev = 1 makes this the last step (x_out = x0).  z ~ N(0,1) is drawn
 * in registers from Philox4x32-10 with key = seed and counter
 * (i/4 low word, i/4 high word, step, 0) and Box-Muller on 23-bit uniforms
 * (see cfg_randn), so it costs no memory traffic and is reproducible.  The
 * integer stream is cfg_randn's exactly; the Gaussian transform is evaluated
 * to the accuracy the storage needs: within a few fp32 ulps for fp32
 * storage (as cfg_randn), within 3.2e-6 absolute for bf16 storage (both
 * bf16 types; the result keeps 8 significant bits): ln u from the hardware
 * base-2 logarithm (a short series for u > 1 - 2^-8), sin and cos from the
 * hardware approximations, a bound that holds for every one of the 2^23
 * uniforms (each factor checked against fp64 over all of them).
 * Fused with the rel-MAE of (pred_c, pred_u) and, when st is given, the
 * schedule update for step `step`: one pass reading x, pred_c, pred_u and
 * writing x_out (4n elements of traffic).
 *   x_out, x_in     device, n elements of dtype (may alias);
 *   pred_c, pred_u  device, n elements of dtype (epsilon predictions);
 *   w               finite guidance scale;
 *   abar_t          in (0, 1); abar_prev in (0, 1], with the DDIM radicands
 *                   non-negative for the given eta (else CFG_ERR_INVALID_ARG);
 *   eta             >= 0, finite;
 *   seed, step      Philox key and counter word (step >= 0);
 *   M_out           device double, nullable;  st, sp: see cfg_relmae_reduce.
 * Rounding, by storage type (the exact step: for the given inputs, the
 * coefficients formed in fp64 on the host, and the drawn z):
 *   CFG_BF16        fp32 arithmetic rounded once to bf16: within one bf16
 *                   ulp of the exact step, equal to its correct rounding
 *                   except where the fp32 evaluation error crosses a
 *                   rounding midpoint;
 *   CFG_BF16_EXACT  the same fp32 evaluation with a per-element error bound;
 *                   the few elements (a few per thousand) whose result lies
 *                   within that bound of a bf16 rounding midpoint are
 *                   recomputed: without noise as the pages write the step,
 *                   in fp64 one correctly rounded operation at a time
 *                   (e = u + w (c - u); x0 = (x - sqrt(1 - abar_t) e) /
 *                   sqrt(abar_t); sqrt(abar_prev) x0 + sqrt(1 - abar_prev) e,
 *                   or x0 on the last step), with noise in double-fp32
 *                   (about 2^-44 of the step's terms); so every element is
 *                   what an fp64 evaluation of the step rounded once to bf16
 *                   gives (without noise: exactly that);
 *   CFG_F32         double-fp32 arithmetic rounded once: the fp32 value
 *                   nearest the exact step in all but rare near-tie cases.
 */
CFG_API int cfg_ddim_step(void* x_out, const void* x_in, const void* pred_c, const void* pred_u,
                          int64_t n, int32_t dtype, float w, double abar_t, double abar_prev,
                          float eta, uint64_t seed, int32_t step, double* M_out,
                          cfg_sched_state* st, const cfg_sched_params* sp, void* ws,
                          size_t ws_bytes, void* stream);

/*
 * cfg_ddim_step without a caller-supplied workspace, for callers that cannot
 * allocate device memory: code running where cudaMalloc is unavailable or
 * forbidden (inside a host framework that owns every device allocation, a
 * plugin or real-time path that must not allocate after start-up, an
 * allocator-free embedding).  No counterpart on the source pages: it is a
 * deployment convenience of this library, not part of the method.
 *
 * Arguments, results and errors are those of cfg_ddim_step, minus ws and
 * ws_bytes.  The scratch is one static device array inside this library of
 * cfg_workspace_bytes() = 196,864 bytes (the maximum: one workspace), held
 * by every GPU that loads the library until the process exits.  No n needs
 * more: the streaming grid is capped at the 4096 block partials one
 * workspace holds, so no size is rejected for want of scratch (n < 0 is
 * rejected as by cfg_ddim_step).  CFG_SCHED_DEFER is rejected
 * (CFG_ERR_INVALID_ARG): every call finishes its rel-MAE in-launch.
 *   - No allocation: the call uses no cudaMalloc, cudaFree, memset or
 *     allocating library routine.
 *   - Set-up: the first call on each device (with that device current) looks
 *     up the array's device address with cudaGetSymbolAddress and caches it
 *     (safe when several host threads make their first call at once); make
 *     that first call before any stream capture.  Nothing is written: the
 *     array is zero when the library's device code loads, and every call
 *     leaves its header (completion counter, no pending work) as it found it.
 *   - Sharing: all calls on a device share the one array, which keeps the
 *     last call's contents.  Calls that may overlap on the GPU (different
 *     streams, or host threads without ordering) race on it: serialise them
 *     on one stream.  Calls in a row on one stream are ordered and may be
 *     issued without host synchronisation between them.
 */
CFG_API int cfg_ddim_step_static_ws(void* x_out, const void* x_in, const void* pred_c,
                                    const void* pred_u, int64_t n, int32_t dtype, float w,
                                    double abar_t, double abar_prev, float eta, uint64_t seed,
                                    int32_t step, double* M_out, cfg_sched_state* st,
                                    const cfg_sched_params* sp, void* stream);

/*
 * One fused CFG + Euler flow step (flow matching, Hybridiff notes "Loss /
 * training strategy": rel-MAE on the velocity pair):
 *   v     = v_u + w (v_c - v_u)
 *   x_out = x + (t_next - t_cur) v
 * with the same fused rel-MAE / schedule handling and arguments as
 * cfg_ddim_step (t_cur, t_next finite; the convention x_t = (1-t) x_0 + t x_1,
 * v = x_1 - x_0, integrates from t = 1 to t = 0).
 */
CFG_API int cfg_flow_step(void* x_out, const void* x_in, const void* v_c, const void* v_u,
                          int64_t n, int32_t dtype, float w, double t_cur, double t_next,
                          int32_t step, double* M_out, cfg_sched_state* st,
                          const cfg_sched_params* sp, void* ws, size_t ws_bytes, void* stream);

/*
 * Batched forms: one launch over `batch` samples laid out back to back in
 * every array (sample b is elements [b n, (b+1) n) with n = n_per_sample),
 * each with its OWN rel-MAE and tau1/tau2 schedule -- the batch-level
 * scale-out of the Hybridiff notes ("Loss / training strategy": every two
 * GPUs produce one image, so each image has its own pair of branches and its
 * own phases).  The update of every element is the unbatched step's (the
 * eta noise counter is the element's index in the whole batch, so a batched
 * step writes the same x as cfg_ddim_step over all batch * n elements); only
 * the reduction and the schedule are per sample.
 *   batch              1 .. 65535;
 *   M_out              device, nullable: batch doubles (M_out[b]);
 *   st                 device, nullable: batch consecutive cfg_sched_state
 *                      structs (st[b]); sp (host) applies to every sample;
 *   ws, ws_bytes       batch consecutive workspaces of cfg_workspace_bytes()
 *                      bytes each (ws_bytes >= batch * cfg_workspace_bytes),
 *                      prepared by cfg_workspace_init_batched (or zeroed);
 *   CFG_SCHED_DEFER    works per sample as for the unbatched calls; complete
 *                      pending work with cfg_workspace_flush_batched.
 * The 128-bit vector path additionally needs n_per_sample * element size to
 * be a multiple of 16 bytes; otherwise the call takes the scalar path.
 * Arguments and errors are otherwise those of the unbatched calls.
 */
CFG_API int cfg_relmae_reduce_batched(const void* pred_c, const void* pred_u,
                                      int64_t n_per_sample, int32_t batch, int32_t dtype,
                                      double* M_out, cfg_sched_state* st,
                                      const cfg_sched_params* sp, int32_t step, void* ws,
                                      size_t ws_bytes, void* stream);
CFG_API int cfg_ddim_step_batched(void* x_out, const void* x_in, const void* pred_c,
                                  const void* pred_u, int64_t n_per_sample, int32_t batch,
                                  int32_t dtype, float w, double abar_t, double abar_prev,
                                  float eta, uint64_t seed, int32_t step, double* M_out,
                                  cfg_sched_state* st, const cfg_sched_params* sp, void* ws,
                                  size_t ws_bytes, void* stream);
CFG_API int cfg_flow_step_batched(void* x_out, const void* x_in, const void* v_c,
                                  const void* v_u, int64_t n_per_sample, int32_t batch,
                                  int32_t dtype, float w, double t_cur, double t_next,
                                  int32_t step, double* M_out, cfg_sched_state* st,
                                  const cfg_sched_params* sp, void* ws, size_t ws_bytes,
                                  void* stream);
/* Prepare / flush `batch` consecutive workspaces (see cfg_workspace_init,
 * cfg_workspace_flush); ws_bytes >= batch * cfg_workspace_bytes(...). */
CFG_API int cfg_workspace_init_batched(void* ws, size_t ws_bytes, int32_t batch, void* stream);
CFG_API int cfg_workspace_flush_batched(void* ws, size_t ws_bytes, int32_t batch, void* stream);

/*
 * Record an externally computed rel-MAE value M as step `step` of the
 * schedule (for callers that reduce the discrepancy elsewhere, e.g. from
 * partial sums of a latent split across devices).  Enqueues one tiny
 * kernel on `stream`.  st: device; sp: host (as cfg_relmae_reduce).
 */
CFG_API int cfg_sched_observe(cfg_sched_state* st, const cfg_sched_params* sp, int32_t step,
                              double M, void* stream);

/*
 * Denoiser callback of cfg_sampler_run: must enqueue on `stream` the two
 * predictions for x_t into pred_c / pred_u (n elements of the run's dtype)
 * and return 0, or return non-zero to stop the run (cfg_sampler_run then
 * returns CFG_ERR_CALLBACK).  For DDIM, `timestep` is the training timestep
 * and `t` its abar; for flow, `timestep` is the step index and `t` the time.
 */
typedef int32_t (*cfg_denoise_fn)(void* user, int32_t step, int32_t timestep, double t,
                                  const void* x_t, void* pred_c, void* pred_u, void* stream);

/*
 * A whole CFG sampler run, host loop over steps start_step .. n_steps-1:
 * the callback fills the predictions, then the fused step updates x in
 * place and the schedule on the device.  No host synchronisation inside.
 *   x                      device, n elements: x_T in, x_0 out;
 *   mode                   CFG_MODE_DDIM or CFG_MODE_FLOW;
 *   abar_table, T          DDIM: host table of abar over T training steps;
 *   timesteps              DDIM: host, n_steps entries in [0, T), the
 *                          timestep of each step, noisiest first (see
 *                          cfg_ddim_timesteps); the step after the last uses
 *                          abar = 1 (the last step returns x0);
 *   t_grid                 FLOW: host, n_steps + 1 times, or NULL for the
 *                          uniform grid t_s = 1 - s/n_steps;
 *   w, eta, seed           as cfg_ddim_step (eta unused for FLOW);
 *   fn, user               denoiser callback;
 *   pred_c_buf, pred_u_buf device, n elements each, filled by the callback;
 *   sp, st                 schedule (both required; sp->n_steps == n_steps);
 *   start_step             first step to run (resume from a saved x and st);
 *   ws, ws_bytes           workspace for n elements.
 */
CFG_API int cfg_sampler_run(void* x, int64_t n, int32_t dtype, int32_t mode,
                            const double* abar_table, int32_t T, const int32_t* timesteps,
                            const double* t_grid, int32_t n_steps, float w, float eta,
                            uint64_t seed, cfg_denoise_fn fn, void* user, void* pred_c_buf,
                            void* pred_u_buf, const cfg_sched_params* sp, cfg_sched_state* st,
                            int32_t start_step, void* ws, size_t ws_bytes, void* stream);

/*
 * Branch callback of cfg_sampler_run_branches: must enqueue on `stream` the
 * prediction of one branch for x_t into `pred` (n elements of the run's
 * dtype) -- branch 0: conditional, 1: unconditional -- and return 0, or
 * return non-zero to stop the run.  `timestep` and `t` as cfg_denoise_fn.
 */
typedef int32_t (*cfg_branch_fn)(void* user, int32_t branch, int32_t step, int32_t timestep,
                                 double t, const void* x_t, void* pred, void* stream);

/*
 * cfg_sampler_run in the CFG-parallel form of the xDiT review (section 3,
 * "CFG Parallelism"): the conditional and the unconditional predictions are
 * produced separately -- there on two GPUs and gathered before the
 * scheduler, here on two streams of one GPU (`stream_c`, `stream_u`) and
 * joined by events before each step on `stream`, so the two branches'
 * kernels may run concurrently.  Every step: the branch streams wait for x_t
 * on `stream`, the callback enqueues branch 0 on stream_c and branch 1 on
 * stream_u, and `stream` waits for both before the fused step.  The three
 * streams must differ.  Three events are created and destroyed inside the
 * call (no device memory is allocated).  Arguments, results and errors are
 * otherwise those of cfg_sampler_run.
 */
CFG_API int cfg_sampler_run_branches(void* x, int64_t n, int32_t dtype, int32_t mode,
                                     const double* abar_table, int32_t T, const int32_t* timesteps,
                                     const double* t_grid, int32_t n_steps, float w, float eta,
                                     uint64_t seed, cfg_branch_fn fn, void* user,
                                     void* pred_c_buf, void* pred_u_buf, void* stream_c,
                                     void* stream_u, const cfg_sched_params* sp,
                                     cfg_sched_state* st, int32_t start_step, void* ws,
                                     size_t ws_bytes, void* stream);

/*
 * Standard normal noise, the same stream the DDIM step draws for eta > 0:
 * out[i] = Box-Muller normal of element i from Philox4x32-10 with key
 * (seed low word, seed high word) and counter (i/4 low, i/4 high, step,
 * stream_id); words (0,1) give elements 4q, 4q+1 as (rho cos, rho sin) with
 * rho = sqrt(-2 ln u0), angle 2 pi u1; words (2,3) likewise give 4q+2, 4q+3;
 * u = (2 (r >> 9) + 1) / 2^24.  The DDIM step uses stream_id 0.  The integer
 * stream is exact; the transform is evaluated in fp32 (exact integer range
 * reduction, short series for ln and sin/cos) to within a few fp32 ulps of
 * the exact values (bf16-storage steps use a cheaper transform of the same
 * integers; see cfg_ddim_step).
 *   out: device float, n elements (n >= 0).
 */
CFG_API int cfg_randn(float* out, int64_t n, uint64_t seed, uint32_t step, uint32_t stream_id,
                      void* stream);

/*
 * Host helpers (no device work).
 * cfg_abar_linear: abar[t] = prod_{i<=t} (1 - beta_i), beta linear from
 *   beta_start to beta_end over T steps, sequential fp64 product.
 *   abar_out: host, T doubles; T >= 1; 0 <= beta_start, beta_end < 1.
 * cfg_ddim_timesteps: the DDIM timestep sequence of the zyxy.net sampler,
 *   round(linspace(0, T-1, n_steps)) walked from the largest down
 *   (ties to even).  out: host, n_steps int32; 1 <= n_steps <= T.
 */
CFG_API int cfg_abar_linear(double* abar_out, int32_t T, double beta_start, double beta_end);
CFG_API int cfg_ddim_timesteps(int32_t* out, int32_t n_steps, int32_t T);

/*
 * Adjacent samplers (host helpers, no device work).  The zyxy.net page names
 * the "linear" and "cosine" noise schedules (section 1) and fewer, spaced
 * sampling steps (section 3); these tables feed cfg_sampler_run and the
 * step calls unchanged.
 * cfg_abar_cosine: the cosine schedule of Nichol and Dhariwal ("Improved
 *   denoising diffusion probabilistic models", 2021):
 *   f(t) = cos^2(((t / T) + s) / (1 + s) * pi / 2),
 *   beta_i = min(1 - f(i + 1) / f(i), max_beta),
 *   abar[i] = prod_{j<=i} (1 - beta_j), sequential fp64 product.
 *   abar_out: host, T doubles; T >= 1; s >= 0 finite (0.008 in the paper);
 *   0 < max_beta < 1 (0.999 in the paper).
 * cfg_timesteps: n_steps training timesteps, noisiest first, by `spacing`:
 *   CFG_SPACING_LINSPACE  round(linspace(0, T-1, n_steps)) (cfg_ddim_timesteps);
 *   CFG_SPACING_LEADING   i * (T / n_steps) (integer ratio), i = n_steps-1 .. 0;
 *   CFG_SPACING_TRAILING  round(T - i * T / n_steps) - 1, i = 0 .. n_steps-1
 *                         (ties to even), so the first step is T - 1.
 *   out: host, n_steps int32; 1 <= n_steps <= T.
 */
enum cfg_spacing { CFG_SPACING_LINSPACE = 0, CFG_SPACING_LEADING = 1, CFG_SPACING_TRAILING = 2 };
CFG_API int cfg_abar_cosine(double* abar_out, int32_t T, double s, double max_beta);
CFG_API int cfg_timesteps(int32_t* out, int32_t n_steps, int32_t T, int32_t spacing);

/*
 * Page-locked host memory for the host<->device copies around a step
 * (cudaHostAlloc, portable to every device).  A step whose inputs and
 * results live in host memory copies 4n elements per step; from buffers
 * allocated here those copies run asynchronously (cfg_copy_async).
 *   cfg_host_alloc: bytes >= 1; *out receives the pointer (host memory,
 *     owned by the caller until cfg_host_free); CFG_ERR_CUDA if the
 *     allocation fails (*out is then NULL).
 *   cfg_host_free: p from cfg_host_alloc, or NULL (a no-op).
 */
CFG_API int cfg_host_alloc(size_t bytes, void** out);
CFG_API int cfg_host_free(void* p);

/*
 * Asynchronous copy of `bytes` bytes between any two of host and device
 * memory (cudaMemcpyAsync, direction from the pointers) on `stream`.  With a
 * page-locked host side (cfg_host_alloc) it returns at once and the copy
 * runs in stream order, overlapping other streams' work; with pageable host
 * memory the CUDA driver stages it and the call may block.
 *   dst, src: non-NULL unless bytes == 0 (then a no-op); the ranges must not
 *   overlap.  CFG_ERR_CUDA if the runtime rejects the copy.
 */
CFG_API int cfg_copy_async(void* dst, const void* src, size_t bytes, void* stream);

/* Message of the last failed call on this host thread ("" if none). */
CFG_API const char* cfg_last_error(void);

/* Library version string. */
CFG_API const char* cfg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CFGSTEP_H */
