// cfgstep_host.cpp -- host-side parts of the CFG sampler-step library: the
// noise-schedule and timestep tables, and the sampler loops that drive the
// fused step of cfgstep.cu through the C ABI (no device code here).
//
// Tables: the linear-beta schedule and the DDIM timestep rule of the zyxy.net
// page ("AIGC text-to-image: how to speed up diffusion-model inference",
// sections 1 and 3), and the adjacent samplers it names (a cosine schedule,
// fewer spaced steps).  Loops: a whole CFG sampler run, with the two branch
// predictions from one callback or from two streams (the CFG-parallel form of
// the xDiT review, section 3).  Page-locked host buffers for the copies around
// a step.

#include <cuda_runtime.h>

#include <math.h>
#include <stdint.h>

#include "cfgstep.h"
#include "cfgstep_internal.h"

using cfgstep::cuda_fail;
using cfgstep::fail;

namespace {

int check_dtype(int32_t dtype) {
  if (dtype != CFG_F32 && dtype != CFG_BF16 && dtype != CFG_BF16_EXACT)
    return fail(CFG_ERR_UNSUPPORTED_DTYPE,
                "unsupported dtype %d (CFG_F32=0, CFG_BF16=1, CFG_BF16_EXACT=2)", dtype);
  return CFG_OK;
}

}  // namespace

extern "C" {

CFG_API int cfg_host_alloc(size_t bytes, void** out) {
  if (out == nullptr) return fail(CFG_ERR_INVALID_ARG, "out must not be NULL");
  *out = nullptr;
  if (bytes == 0) return fail(CFG_ERR_INVALID_ARG, "bytes must be >= 1");
  const cudaError_t e = cudaHostAlloc(out, bytes, cudaHostAllocPortable);
  if (e != cudaSuccess) {
    *out = nullptr;
    return cuda_fail(e, "cudaHostAlloc");
  }
  return CFG_OK;
}

CFG_API int cfg_host_free(void* p) {
  if (p == nullptr) return CFG_OK;
  const cudaError_t e = cudaFreeHost(p);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFreeHost");
  return CFG_OK;
}

CFG_API int cfg_copy_async(void* dst, const void* src, size_t bytes, void* stream) {
  if (bytes == 0) return CFG_OK;
  if (dst == nullptr || src == nullptr) return fail(CFG_ERR_INVALID_ARG, "dst and src must not be NULL");
  const cudaError_t e =
      cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
  return CFG_OK;
}

CFG_API int cfg_abar_linear(double* abar_out, int32_t T, double beta_start, double beta_end) {
  if (abar_out == nullptr) return fail(CFG_ERR_INVALID_ARG, "abar_out must not be NULL");
  if (T < 1) return fail(CFG_ERR_INVALID_ARG, "T must be >= 1");
  if (!(beta_start >= 0.0 && beta_start < 1.0 && beta_end >= 0.0 && beta_end < 1.0))
    return fail(CFG_ERR_INVALID_ARG, "betas must be in [0, 1)");
  // beta_i = beta_start + i * (beta_end - beta_start) / (T - 1), the last one exactly beta_end.
  const double step = T > 1 ? (beta_end - beta_start) / static_cast<double>(T - 1) : 0.0;
  double acc = 1.0;
  for (int32_t i = 0; i < T; ++i) {
    const double beta = (T > 1 && i == T - 1) ? beta_end : static_cast<double>(i) * step + beta_start;
    acc = acc * (1.0 - beta);
    abar_out[i] = acc;
  }
  return CFG_OK;
}

CFG_API int cfg_ddim_timesteps(int32_t* out, int32_t n_steps, int32_t T) {
  if (out == nullptr) return fail(CFG_ERR_INVALID_ARG, "out must not be NULL");
  if (T < 1 || n_steps < 1 || n_steps > T)
    return fail(CFG_ERR_INVALID_ARG, "need 1 <= n_steps <= T (got n_steps=%d, T=%d)", n_steps, T);
  const double step = n_steps > 1 ? static_cast<double>(T - 1) / static_cast<double>(n_steps - 1) : 0.0;
  for (int32_t j = 0; j < n_steps; ++j) {
    const double v = (n_steps > 1 && j == n_steps - 1) ? static_cast<double>(T - 1)
                                                       : static_cast<double>(j) * step;
    out[n_steps - 1 - j] = static_cast<int32_t>(nearbyint(v));  // ties to even
  }
  return CFG_OK;
}

CFG_API int cfg_abar_cosine(double* abar_out, int32_t T, double s, double max_beta) {
  if (abar_out == nullptr) return fail(CFG_ERR_INVALID_ARG, "abar_out must not be NULL");
  if (T < 1) return fail(CFG_ERR_INVALID_ARG, "T must be >= 1");
  if (!(s >= 0.0 && isfinite(s))) return fail(CFG_ERR_INVALID_ARG, "s must be finite and >= 0");
  if (!(max_beta > 0.0 && max_beta < 1.0))
    return fail(CFG_ERR_INVALID_ARG, "max_beta must be in (0, 1)");
  const double half_pi = 1.57079632679489661923;
  auto f = [&](int32_t t) {
    const double c = cos((static_cast<double>(t) / static_cast<double>(T) + s) / (1.0 + s) * half_pi);
    return c * c;
  };
  double acc = 1.0, f_prev = f(0);
  for (int32_t i = 0; i < T; ++i) {
    const double f_next = f(i + 1);
    double beta = 1.0 - f_next / f_prev;
    if (beta > max_beta) beta = max_beta;
    acc = acc * (1.0 - beta);
    abar_out[i] = acc;
    f_prev = f_next;
  }
  return CFG_OK;
}

CFG_API int cfg_timesteps(int32_t* out, int32_t n_steps, int32_t T, int32_t spacing) {
  if (spacing == CFG_SPACING_LINSPACE) return cfg_ddim_timesteps(out, n_steps, T);
  if (out == nullptr) return fail(CFG_ERR_INVALID_ARG, "out must not be NULL");
  if (T < 1 || n_steps < 1 || n_steps > T)
    return fail(CFG_ERR_INVALID_ARG, "need 1 <= n_steps <= T (got n_steps=%d, T=%d)", n_steps, T);
  if (spacing == CFG_SPACING_LEADING) {
    const int32_t ratio = T / n_steps;
    for (int32_t i = 0; i < n_steps; ++i) out[i] = (n_steps - 1 - i) * ratio;
    return CFG_OK;
  }
  if (spacing == CFG_SPACING_TRAILING) {
    const double step = static_cast<double>(T) / static_cast<double>(n_steps);
    for (int32_t i = 0; i < n_steps; ++i)
      out[i] = static_cast<int32_t>(nearbyint(static_cast<double>(T) - static_cast<double>(i) * step)) - 1;
    return CFG_OK;
  }
  return fail(CFG_ERR_INVALID_ARG, "unknown spacing %d", spacing);
}

}  // extern "C"

namespace {

// Where a run's predictions come from: one callback that fills both on the
// run's stream, or (the CFG-parallel form of the xDiT review, section 3) one
// callback per branch, each on its own stream, joined by events before the
// step -- on one GPU the two branches' kernels may overlap.
struct Producer {
  cfg_denoise_fn both = nullptr;
  cfg_branch_fn branch = nullptr;
  void* user = nullptr;
  cudaStream_t sc = nullptr, su = nullptr;
  cudaEvent_t ready = nullptr, done_c = nullptr, done_u = nullptr;

  // Enqueue the two predictions of step s; returns the callback's status in *cb.
  int produce(int32_t s, int32_t timestep, double t, void* x, void* pc, void* pu,
              cudaStream_t stream, int32_t* cb) {
    if (both) {
      *cb = both(user, s, timestep, t, x, pc, pu, stream);
      return CFG_OK;
    }
    cudaError_t e = cudaEventRecord(ready, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(sc, ready, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(su, ready, 0);
    if (e != cudaSuccess) return cuda_fail(e, "branch stream fork");
    *cb = branch(user, 0, s, timestep, t, x, pc, sc);
    if (*cb == 0) *cb = branch(user, 1, s, timestep, t, x, pu, su);
    e = cudaEventRecord(done_c, sc);
    if (e == cudaSuccess) e = cudaEventRecord(done_u, su);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, done_c, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, done_u, 0);
    if (e != cudaSuccess) return cuda_fail(e, "branch stream join");
    return CFG_OK;
  }
};

int run_loop(void* x, int64_t n, int32_t dtype, int32_t mode, const double* abar_table, int32_t T,
             const int32_t* timesteps, const double* t_grid, int32_t n_steps, float w, float eta,
             uint64_t seed, Producer& prod, void* pred_c_buf, void* pred_u_buf,
             const cfg_sched_params* sp, cfg_sched_state* st, int32_t start_step, void* ws,
             size_t ws_bytes, void* stream) {
  if (st == nullptr || sp == nullptr)
    return fail(CFG_ERR_INVALID_ARG, "schedule state and parameters are required");
  if (n_steps < 1 || n_steps > CFG_SCHED_MAX_STEPS)
    return fail(CFG_ERR_INVALID_ARG, "n_steps must be in [1, %d]", CFG_SCHED_MAX_STEPS);
  if (sp->n_steps != n_steps)
    return fail(CFG_ERR_INVALID_ARG, "sp->n_steps (%d) != n_steps (%d)", sp->n_steps, n_steps);
  if (start_step < 0 || start_step > n_steps)
    return fail(CFG_ERR_INVALID_ARG, "start_step must be in [0, n_steps]");
  if (n > 0 && (x == nullptr || pred_c_buf == nullptr || pred_u_buf == nullptr))
    return fail(CFG_ERR_INVALID_ARG, "x and prediction buffers must not be NULL");
  int rc = check_dtype(dtype);
  if (rc) return rc;
  if (mode == CFG_MODE_DDIM) {
    if (abar_table == nullptr || timesteps == nullptr || T < 1)
      return fail(CFG_ERR_INVALID_ARG, "DDIM needs abar_table, T >= 1 and timesteps");
    for (int32_t s = 0; s < n_steps; ++s)
      if (timesteps[s] < 0 || timesteps[s] >= T)
        return fail(CFG_ERR_INVALID_ARG, "timesteps[%d] = %d outside [0, %d)", s, timesteps[s], T);
  } else if (mode != CFG_MODE_FLOW) {
    return fail(CFG_ERR_INVALID_ARG, "unknown mode %d", mode);
  }
  const cudaStream_t cs = static_cast<cudaStream_t>(stream);
  // Whole runs defer each step's reduction to the next step's launch; the
  // last step finishes in-launch, so the state is complete when the run is.
  cfg_sched_params run_sp = *sp;
  run_sp.flags |= CFG_SCHED_DEFER;
  int32_t cb = 0, failed_step = -1;
  for (int32_t s = start_step; s < n_steps; ++s) {
    if (mode == CFG_MODE_DDIM) {
      const double ab = abar_table[timesteps[s]];
      const double ab_prev = (s + 1 < n_steps) ? abar_table[timesteps[s + 1]] : 1.0;
      rc = prod.produce(s, timesteps[s], ab, x, pred_c_buf, pred_u_buf, cs, &cb);
      if (rc) return rc;
      if (cb != 0) {
        failed_step = s;
        break;
      }
      rc = cfg_ddim_step(x, x, pred_c_buf, pred_u_buf, n, dtype, w, ab, ab_prev, eta, seed, s,
                         nullptr, st, &run_sp, ws, ws_bytes, cs);
    } else {
      const double t = t_grid ? t_grid[s] : 1.0 - static_cast<double>(s) / n_steps;
      const double tn = t_grid ? t_grid[s + 1] : 1.0 - static_cast<double>(s + 1) / n_steps;
      rc = prod.produce(s, s, t, x, pred_c_buf, pred_u_buf, cs, &cb);
      if (rc) return rc;
      if (cb != 0) {
        failed_step = s;
        break;
      }
      rc = cfg_flow_step(x, x, pred_c_buf, pred_u_buf, n, dtype, w, t, tn, s, nullptr, st, &run_sp,
                         ws, ws_bytes, cs);
    }
    if (rc) return rc;
  }
  if (cb != 0) {
    // complete the last finished step before reporting the callback's error
    rc = cfg_workspace_flush(ws, ws_bytes, stream);
    if (rc) return rc;
    return fail(CFG_ERR_CALLBACK, "denoiser callback returned %d at step %d", cb, failed_step);
  }
  return CFG_OK;
}

}  // namespace

extern "C" {

CFG_API int cfg_sampler_run(void* x, int64_t n, int32_t dtype, int32_t mode,
                            const double* abar_table, int32_t T, const int32_t* timesteps,
                            const double* t_grid, int32_t n_steps, float w, float eta,
                            uint64_t seed, cfg_denoise_fn fn, void* user, void* pred_c_buf,
                            void* pred_u_buf, const cfg_sched_params* sp, cfg_sched_state* st,
                            int32_t start_step, void* ws, size_t ws_bytes, void* stream) {
  if (fn == nullptr) return fail(CFG_ERR_INVALID_ARG, "denoiser callback must not be NULL");
  Producer prod;
  prod.both = fn;
  prod.user = user;
  return run_loop(x, n, dtype, mode, abar_table, T, timesteps, t_grid, n_steps, w, eta, seed, prod,
                  pred_c_buf, pred_u_buf, sp, st, start_step, ws, ws_bytes, stream);
}

CFG_API int cfg_sampler_run_branches(void* x, int64_t n, int32_t dtype, int32_t mode,
                                     const double* abar_table, int32_t T, const int32_t* timesteps,
                                     const double* t_grid, int32_t n_steps, float w, float eta,
                                     uint64_t seed, cfg_branch_fn fn, void* user,
                                     void* pred_c_buf, void* pred_u_buf, void* stream_c,
                                     void* stream_u, const cfg_sched_params* sp,
                                     cfg_sched_state* st, int32_t start_step, void* ws,
                                     size_t ws_bytes, void* stream) {
  if (fn == nullptr) return fail(CFG_ERR_INVALID_ARG, "branch callback must not be NULL");
  if (stream_c == stream || stream_u == stream || stream_c == stream_u)
    return fail(CFG_ERR_INVALID_ARG, "the two branch streams and the run's stream must differ");
  Producer prod;
  prod.branch = fn;
  prod.user = user;
  prod.sc = static_cast<cudaStream_t>(stream_c);
  prod.su = static_cast<cudaStream_t>(stream_u);
  cudaEvent_t* evs[3] = {&prod.ready, &prod.done_c, &prod.done_u};
  int rc = CFG_OK;
  for (cudaEvent_t* ev : evs) {
    const cudaError_t e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      rc = cuda_fail(e, "cudaEventCreateWithFlags");
      break;
    }
  }
  if (rc == CFG_OK)
    rc = run_loop(x, n, dtype, mode, abar_table, T, timesteps, t_grid, n_steps, w, eta, seed, prod,
                  pred_c_buf, pred_u_buf, sp, st, start_step, ws, ws_bytes, stream);
  for (cudaEvent_t* ev : evs)
    if (*ev) cudaEventDestroy(*ev);
  return rc;
}

}  // extern "C"
