"""CPU oracle of the classifier-free-guidance sampler step (fp64, NumPy).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import
this module.  It shares no code with the CUDA library and never imports it.

Plain and slow on purpose: every function is the definition written out in
float64, vectorised with NumPy elementwise operations and ``np.sum`` only.
Stored tensors (fp32, or bf16 bit patterns) are widened exactly to float64;
each output the method stores is rounded once to the storage type (fp32:
IEEE round-to-nearest-even; bf16: round-to-nearest-even of the exact fp64
value).  A storage type "f64" turns rounding off (used by the pins that
check the mathematics against closed forms).

Sources (the pages the method is defined on):

* [HYB] "Accelerating Diffusion via Hybrid Data-Pipeline Parallelism Based on
  Conditional Guidance Scheduling" (CVPR 2026 paper notes, papernotes.org):
  - "Method / Overall framework": two branches, three phases
    Warm-Up [T, tau1], Parallelism (tau1, tau2), Fully-Connecting [tau2, 0];
  - "Key design 2": the denoising discrepancy rel-MAE between the two noise
    predictions (its formula is lost in the page's extraction; the L1-ratio
    form of its score decomposition fixes the reading used here);
  - "Key design 3": slope G_t = (M_t - M_{t-L}) / L, tau1' = first t with
    0 <= G_t < g_slope, tau1 = min(tau1', tau_cap) with tau_cap the global
    minimum of the discrepancy curve, tau2 = tau1 + k;
  - "Loss / training strategy": flow-matching models use the velocity pair
    (v_c, v_u) in place of the noise pair.
* [ZYX] "AIGC text-to-image: how to speed up diffusion-model inference"
  (zyxy.net), section 3 "Algorithm-level optimisation", the DDIM sampler:
  timestep sequence linspace(0, T-1, N) rounded and walked in reverse;
  sigma_eta, the x0 prediction, the DDIM update with sigma_eta * noise, and
  the last step returning the x0 prediction.
* [XDIT] xDiT review, section 3 "CFG Parallelism": the conditional and
  unconditional predictions are gathered before the scheduler runs; the
  scheduler call is the step computed here.

Readings where the pages are silent or garbled (each also listed in the
design notes):

* guidance: e = e_u + w (e_c - e_u) (w = 1 gives the conditional branch);
* rel-MAE: sum|e_c - e_u| / sum|e_u| over the whole latent (a ratio of
  means); 0/0 -> 0 and x/0 -> +inf;
* the "t" of the schedule rule is the step index s counted from the first
  denoising step; G_s exists for s >= L; tau_cap = earliest argmin of the
  run's own trace unless a calibrated cap >= 0 is given; NaN compares false;
* the x0 prediction uses sqrt(1 - abar_t) as the noise scale (the only
  reading under which the page's update is DDIM); the generic loop's update
  in section 1 of [ZYX] is not DDIM and is not used;
* the last DDIM step returns x0 (the page's last-step branch);
* flow matching: x_t = (1 - t) x_0 + t x_1, v = x_1 - x_0, Euler on a uniform
  grid t_i = 1 - i/N;
* eta noise: Philox4x32-10 (Salmon et al., SC'11) keyed by the seed with
  counter (element/4 low, high, step, stream 0), Box-Muller on 23-bit
  uniforms (2k+1)/2^24 (exact in fp32).
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Callable, Dict, List, Optional, Tuple

import numpy as np

TAU_NONE = 2**31 - 1          # "undefined / never" for tau values
PHASE_WARMUP, PHASE_PARALLEL, PHASE_FULL = 0, 1, 2

# ---------------------------------------------------------------------------
# Storage rounding
# ---------------------------------------------------------------------------
BF16_MAX = float.fromhex("0x1.fep127")


def round_bf16(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value, ties to even.

    bf16 keeps 8 significant bits.  For |v| in [2^e, 2^(e+1)) the spacing is
    2^(e-7); below 2^-126 (subnormals) it is 2^-133.  The value is scaled by
    a power of two (exact), rounded half-to-even to an integer, scaled back.
    Values whose rounded magnitude exceeds the largest bf16 become +-inf.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.array(v, copy=True)
    fin = np.isfinite(v) & (v != 0.0)
    _, e = np.frexp(v[fin])                 # v = m * 2^e, 0.5 <= |m| < 1
    q = np.maximum(e - 8, -133)             # spacing exponent
    r = np.ldexp(np.round(np.ldexp(v[fin], -q)), q)
    r = np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, r), r)
    out[fin] = r
    return out


def round_f32(v: np.ndarray) -> np.ndarray:
    """Round float64 values to fp32 (IEEE nearest even) and widen back."""
    return np.asarray(v, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_storage(v: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f64":
        return np.asarray(v, dtype=np.float64)
    if dtype == "f32":
        return round_f32(v)
    if dtype == "bf16":
        return round_bf16(v)
    raise ValueError(dtype)


def f32_bits_to_bf16_bits(b: np.ndarray) -> np.ndarray:
    """fp32 bit patterns -> bf16 bit patterns, round to nearest even (NaN -> quiet NaN)."""
    b = np.asarray(b, dtype=np.uint32)
    nan = (b & 0x7FFFFFFF) > 0x7F800000
    r = ((b + np.uint32(0x7FFF) + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    return np.where(nan, np.uint16(0x7FC0), r).astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Bit patterns of round_bf16(v) (the value is exact in fp32, so take its top half)."""
    r = round_bf16(v).astype(np.float32)
    return (r.view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# Noise schedule and timesteps
# ---------------------------------------------------------------------------
def abar_linear(T: int = 1000, beta_start: float = 1e-4, beta_end: float = 0.02) -> np.ndarray:
    """abar_t = prod_{i<=t} (1 - beta_i), beta linear from beta_start to beta_end.

    [ZYX] section 1 names a linear schedule; the range is the workload's.
    The product is taken sequentially in float64.
    """
    betas = np.linspace(beta_start, beta_end, T, dtype=np.float64)
    abar = np.empty(T, dtype=np.float64)
    acc = 1.0
    for i in range(T):
        acc = acc * (1.0 - betas[i])
        abar[i] = acc
    return abar


def ddim_timesteps(N: int, T: int = 1000) -> np.ndarray:
    """[ZYX] DDIM: linspace(0, T-1, N) rounded to integers, walked from the largest down."""
    seq = np.linspace(0, T - 1, N).round().astype(np.int64)
    return seq[::-1].copy()


def abar_cosine(T: int = 1000, s: float = 0.008, max_beta: float = 0.999) -> np.ndarray:
    """[ZYX] section 1 names a cosine schedule; its definition (reading) is Nichol and
    Dhariwal's: abar(t) = f(t)/f(0) with f(t) = cos^2(((t/T) + s)/(1 + s) * pi/2), applied
    through beta_i = 1 - f(i+1)/f(i) clipped at max_beta, abar_i = prod_{j<=i} (1 - beta_j)
    (sequential fp64 product)."""
    def f(t):
        return math.cos((t / T + s) / (1.0 + s) * math.pi / 2.0) ** 2
    abar = np.empty(T, dtype=np.float64)
    acc = 1.0
    for i in range(T):
        beta = min(1.0 - f(i + 1) / f(i), max_beta)
        acc = acc * (1.0 - beta)
        abar[i] = acc
    return abar


def timesteps(N: int, T: int = 1000, spacing: str = "linspace") -> np.ndarray:
    """N training timesteps, noisiest first.  "linspace" is the [ZYX] DDIM rule; "leading"
    (i * (T // N)) and "trailing" (round(T - i T/N) - 1, which starts at T - 1) are the
    spacings of Lin et al. 2023 ("Common diffusion noise schedules and sample steps are
    flawed") for fewer, spaced steps ([ZYX] section 3)."""
    if spacing == "linspace":
        return ddim_timesteps(N, T)
    if spacing == "leading":
        return (np.arange(N, dtype=np.int64) * (T // N))[::-1].copy()
    if spacing == "trailing":
        return np.array([int(np.round(T - i * (T / N))) - 1 for i in range(N)], dtype=np.int64)
    raise ValueError(spacing)


def flow_times(N: int) -> np.ndarray:
    """Uniform Euler grid on t in [1, 0]: t_i = 1 - i/N, i = 0..N (reading)."""
    return np.array([1.0 - i / N for i in range(N + 1)], dtype=np.float64)


# ---------------------------------------------------------------------------
# The step
# ---------------------------------------------------------------------------
def rel_mae(pred_c: np.ndarray, pred_u: np.ndarray) -> float:
    """[HYB] key design 2: M = mean|e_c - e_u| / mean|e_u| over the whole latent.

    Equal n cancels, so this is sum|e_c - e_u| / sum|e_u|.  0/0 -> 0 (no
    discrepancy between identical zero predictions); x/0 -> +inf.
    """
    c = np.asarray(pred_c, dtype=np.float64)
    u = np.asarray(pred_u, dtype=np.float64)
    s_diff = float(np.sum(np.abs(c - u)))
    s_u = float(np.sum(np.abs(u)))
    if s_u == 0.0:
        if math.isnan(s_diff):
            return math.nan
        return 0.0 if s_diff == 0.0 else math.inf
    return s_diff / s_u


def rel_mae_per_sample(pred_c: np.ndarray, pred_u: np.ndarray, batch: int) -> np.ndarray:
    """[HYB] loss/training strategy, batch-level scale-out: every image is produced by its own
    pair of branches, so each of the ``batch`` samples (equal consecutive slices of the latent)
    has its own discrepancy M_b = rel_mae(sample b's predictions)."""
    c = np.asarray(pred_c, dtype=np.float64).reshape(batch, -1)
    u = np.asarray(pred_u, dtype=np.float64).reshape(batch, -1)
    return np.array([rel_mae(c[b], u[b]) for b in range(batch)], dtype=np.float64)


def guidance(pred_c: np.ndarray, pred_u: np.ndarray, w: float) -> np.ndarray:
    """Classifier-free guidance: e = e_u + w (e_c - e_u)."""
    c = np.asarray(pred_c, dtype=np.float64)
    u = np.asarray(pred_u, dtype=np.float64)
    return u + w * (c - u)


def ddim_sigma(abar_t: float, abar_prev: float, eta: float) -> float:
    """[ZYX] DDIM: sigma_eta = eta sqrt((1 - abar_prev)/(1 - abar_t) (1 - abar_t/abar_prev))."""
    return eta * math.sqrt((1.0 - abar_prev) / (1.0 - abar_t) * (1.0 - abar_t / abar_prev))


def ddim_update(x: np.ndarray, e: np.ndarray, abar_t: float, abar_prev: float, eta: float,
                z: Optional[np.ndarray], last: bool) -> np.ndarray:
    """[ZYX] DDIM update on float64 arrays.

    x0 = (x - sqrt(1 - abar_t) e) / sqrt(abar_t);
    not last: x_prev = sqrt(abar_prev) x0 + sqrt(1 - abar_prev - sigma^2) e + sigma z;
    last: x_prev = x0.
    """
    x = np.asarray(x, dtype=np.float64)
    e = np.asarray(e, dtype=np.float64)
    x0 = (x - math.sqrt(1.0 - abar_t) * e) / math.sqrt(abar_t)
    if last:
        return x0
    sigma = ddim_sigma(abar_t, abar_prev, eta)
    dir_sq = 1.0 - abar_prev - sigma * sigma
    if dir_sq < 0.0:
        if dir_sq < -1e-12:
            raise ValueError("eta too large: 1 - abar_prev - sigma^2 < 0")
        dir_sq = 0.0
    out = math.sqrt(abar_prev) * x0 + math.sqrt(dir_sq) * e
    if sigma != 0.0:
        out = out + sigma * np.asarray(z, dtype=np.float64)
    return out


def euler_update(x: np.ndarray, v: np.ndarray, t_cur: float, t_next: float) -> np.ndarray:
    """Euler step of the flow ODE dx/dt = v from t_cur to t_next."""
    return np.asarray(x, dtype=np.float64) + (t_next - t_cur) * np.asarray(v, dtype=np.float64)


# ---------------------------------------------------------------------------
# Philox4x32-10 and the Gaussian transform
# ---------------------------------------------------------------------------
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
_MASK32 = 0xFFFFFFFF


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Philox4x32 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC'11).

    One round maps counter words (X0, X1, X2, X3) and key (K0, K1) to
    (hi(M1*X2) ^ X1 ^ K0, lo(M1*X2), hi(M0*X0) ^ X3 ^ K1, lo(M0*X0));
    between rounds the key is bumped by the Weyl constants (W0, W1).
    Arrays of uint32 in, four arrays of uint32 out.
    """
    x0 = np.asarray(c0, dtype=np.uint64) & _MASK32
    x1 = np.asarray(c1, dtype=np.uint64) & _MASK32
    x2 = np.asarray(c2, dtype=np.uint64) & _MASK32
    x3 = np.asarray(c3, dtype=np.uint64) & _MASK32
    k0 = int(k0) & _MASK32
    k1 = int(k1) & _MASK32
    m0 = np.uint64(PHILOX_M0)
    m1 = np.uint64(PHILOX_M1)
    for rnd in range(10):
        p0 = x0 * m0                      # < 2^64, exact in uint64
        p1 = x2 * m1
        hi0, lo0 = p0 >> np.uint64(32), p0 & np.uint64(_MASK32)
        hi1, lo1 = p1 >> np.uint64(32), p1 & np.uint64(_MASK32)
        x0, x1, x2, x3 = (hi1 ^ x1 ^ np.uint64(k0), lo1, hi0 ^ x3 ^ np.uint64(k1), lo0)
        k0 = (k0 + PHILOX_W0) & _MASK32
        k1 = (k1 + PHILOX_W1) & _MASK32
    return tuple(a.astype(np.uint32) for a in (x0, x1, x2, x3))


def uniform_from_bits(r: np.ndarray) -> np.ndarray:
    """23-bit uniform on (0,1): (2 * (r >> 9) + 1) / 2^24 (exact in fp32 and fp64)."""
    k = (np.asarray(r, dtype=np.uint32) >> 9).astype(np.float64)
    return (2.0 * k + 1.0) / 16777216.0


def gaussian_noise(n: int, seed: int, step: int, stream: int = 0, start: int = 0) -> np.ndarray:
    """N(0,1) noise for elements start .. start+n-1 of one step.

    Element i uses Philox block q = i // 4 with counter (q mod 2^32,
    q >> 32, step, stream) and key (seed mod 2^32, seed >> 32); word
    j = i % 4.  Box-Muller on the word pairs: with u_a = uniform(w0),
    u_b = uniform(w1), rho = sqrt(-2 ln u_a):
      word 0 -> rho cos(2 pi u_b), word 1 -> rho sin(2 pi u_b),
    and words 2, 3 likewise from (w2, w3).
    """
    idx = np.arange(start, start + n, dtype=np.int64)
    q = idx // 4
    j = idx % 4
    qb = np.unique(q)
    w = philox4x32_10(qb & _MASK32, qb >> 32, np.full(qb.shape, step & _MASK32),
                      np.full(qb.shape, stream & _MASK32), seed & _MASK32, (seed >> 32) & _MASK32)
    u = [uniform_from_bits(wi) for wi in w]
    rho01 = np.sqrt(-2.0 * np.log(u[0]))
    rho23 = np.sqrt(-2.0 * np.log(u[2]))
    th01 = 2.0 * math.pi * u[1]
    th23 = 2.0 * math.pi * u[3]
    z = np.stack([rho01 * np.cos(th01), rho01 * np.sin(th01),
                  rho23 * np.cos(th23), rho23 * np.sin(th23)], axis=1)   # [blocks, 4]
    pos = np.searchsorted(qb, q)
    return z[pos, j]


# ---------------------------------------------------------------------------
# The tau1 / tau2 schedule
# ---------------------------------------------------------------------------
@dataclass
class Schedule:
    tau1p: int
    tau_cap: int
    tau1: int
    tau2: int
    decided_at: int
    G: np.ndarray
    phase: np.ndarray

    def as_dict(self) -> Dict[str, int]:
        return {"tau1p": self.tau1p, "tau_cap": self.tau_cap, "tau1": self.tau1,
                "tau2": self.tau2, "decided_at": self.decided_at}


def schedule(M: np.ndarray, L: int, g_slope: float, k: int, tau_cap: int = -1) -> Schedule:
    """[HYB] key design 3 on a full rel-MAE trace M[0..N-1] (step index s, first step = 0).

    G_s = (M_s - M_{s-L}) / L for s >= L;
    tau1' = first s with 0 <= G_s < g_slope (TAU_NONE if none);
    tau_cap = the calibrated cap if >= 0, else the earliest index of the
    smallest non-NaN M (TAU_NONE if all NaN);
    tau1 = min(tau1', tau_cap); tau2 = tau1 + k (TAU_NONE stays TAU_NONE).
    phase[s] = Warm-Up if s <= tau1, Parallelism if tau1 < s < tau2, else
    Fully-Connecting ([HYB] overall framework).
    decided_at: with a calibrated cap, the step min(tau1', tau_cap) at which
    tau1 is known (capped at N-1); with the trace's own argmin, N-1.
    """
    M = np.asarray(M, dtype=np.float64)
    N = int(M.shape[0])
    G = np.full(N, np.nan)
    tau1p = TAU_NONE
    for s in range(L, N):
        G[s] = (M[s] - M[s - L]) / L
        if tau1p == TAU_NONE and (G[s] >= 0.0) and (G[s] < g_slope):
            tau1p = s
    argmin = -1
    for s in range(N):
        if not math.isnan(M[s]) and (argmin < 0 or M[s] < M[argmin]):
            argmin = s
    if tau_cap >= 0:
        cap = int(tau_cap)
        decided_at = min(min(tau1p, cap), N - 1)
    else:
        cap = argmin if argmin >= 0 else TAU_NONE
        decided_at = N - 1
    tau1 = min(tau1p, cap)
    tau2 = TAU_NONE if tau1 == TAU_NONE else min(tau1 + k, TAU_NONE)
    phase = np.empty(N, dtype=np.uint8)
    for s in range(N):
        phase[s] = PHASE_WARMUP if s <= tau1 else (PHASE_PARALLEL if s < tau2 else PHASE_FULL)
    return Schedule(tau1p, cap, tau1, tau2, decided_at, G, phase)


# ---------------------------------------------------------------------------
# One stored step (what the library's single-step calls compute)
# ---------------------------------------------------------------------------
def ddim_step(x: np.ndarray, pred_c: np.ndarray, pred_u: np.ndarray, dtype: str, w: float,
              abar_t: float, abar_prev: float, eta: float, seed: int, step: int,
              last: bool = False, z: Optional[np.ndarray] = None) -> Tuple[np.ndarray, float]:
    """rel-MAE, guidance and DDIM update on stored float64 values; returns (stored x_prev, M)."""
    M = rel_mae(pred_c, pred_u)
    e = guidance(pred_c, pred_u, w)
    if z is None and eta != 0.0 and not last:
        z = gaussian_noise(np.asarray(x).size, seed, step)
    out = ddim_update(x, e, abar_t, abar_prev, eta, z, last)
    return round_storage(out, dtype), M


def flow_step(x: np.ndarray, pred_c: np.ndarray, pred_u: np.ndarray, dtype: str, w: float,
              t_cur: float, t_next: float) -> Tuple[np.ndarray, float]:
    """rel-MAE on the velocity pair, guidance and Euler update; returns (stored x_next, M)."""
    M = rel_mae(pred_c, pred_u)
    v = guidance(pred_c, pred_u, w)
    return round_storage(euler_update(x, v, t_cur, t_next), dtype), M


# ---------------------------------------------------------------------------
# Synthetic denoisers (the model stand-ins of the workloads)
# ---------------------------------------------------------------------------
def _round_pred(v: np.ndarray, dtype: str) -> np.ndarray:
    """Harness rounding of a denoiser output: fp64 -> fp32 (nearest even) -> storage."""
    if dtype == "f64":
        return v
    v32 = round_f32(v)
    if dtype == "f32":
        return v32
    return bf16_bits_to_f64(f32_bits_to_bf16_bits(v32.astype(np.float32).view(np.uint32)))


def gaussian_eps(x: np.ndarray, mean: np.ndarray, abar: float, std: float,
                 perturb: Optional[np.ndarray], dtype: str) -> np.ndarray:
    """Posterior-mean noise prediction for data N(mean, std^2) (std = 0: a point mass at mean).

    With x_t = sqrt(abar) x_0 + sqrt(1-abar) eps, (eps, x_t) are jointly
    Gaussian and E[eps | x_t] = A (x_t - sqrt(abar) mean) with
    A = sqrt(1-abar) / (abar std^2 + 1 - abar).  Evaluated as
    ((x - sa*mean) * A) (+ perturb), each operation rounded in fp64,
    then rounded fp64 -> fp32 -> storage.
    """
    sa = math.sqrt(abar)
    A = math.sqrt(1.0 - abar) / (abar * std * std + (1.0 - abar))
    t = np.asarray(mean, dtype=np.float64) * sa
    t = np.asarray(x, dtype=np.float64) - t
    t = t * A
    if perturb is not None:
        t = t + np.asarray(perturb, dtype=np.float64)
    return _round_pred(t, dtype)


def flow_velocity(x: np.ndarray, mean: np.ndarray, t: float, dtype: str) -> np.ndarray:
    """Velocity of a point mass at ``mean``: x_t = (1-t) mean + t x_1 gives v = x_1 - mean = (x_t - mean)/t.

    Evaluated as (x - mean) * (1/t) in fp64, then rounded fp64 -> fp32 -> storage.
    """
    inv_t = 1.0 / t
    v = (np.asarray(x, dtype=np.float64) - np.asarray(mean, dtype=np.float64)) * inv_t
    return _round_pred(v, dtype)


# ---------------------------------------------------------------------------
# A whole sampler run on one workload
# ---------------------------------------------------------------------------
@dataclass
class RunResult:
    x0: np.ndarray                 # final stored latent (float64 values)
    M: np.ndarray                  # rel-MAE trace [N]
    sched: Schedule
    trajectory: Optional[List[np.ndarray]] = None
    M_samples: Optional[np.ndarray] = None          # [N, batch] per-sample traces
    sched_samples: Optional[List[Schedule]] = None  # one schedule per sample


def run_sampler(wl, inputs: Dict[str, np.ndarray], perturb: Optional[Callable] = None,
                dtype: Optional[str] = None, keep_trajectory: bool = False,
                w: Optional[float] = None, batch: Optional[int] = None) -> RunResult:
    """The full N-step CFG sampler on a workload (``workloads.Workload``) in float64.

    ``inputs`` comes from ``workloads.draw_inputs``; ``perturb(step, branch)``
    supplies the per-step prediction perturbation (``workloads.draw_perturbation``).
    ``dtype`` overrides the storage type ("f64" turns rounding off).  With ``batch``,
    the per-sample traces M_b and schedules of the batch-level scale-out are recorded too
    (the update of x is the same).
    """
    dt = dtype or wl.dtype
    wv = wl.w if w is None else w
    xT = inputs["x_T"]
    x = bf16_bits_to_f64(xT) if xT.dtype == np.uint16 else np.asarray(xT, dtype=np.float64)
    x = x.reshape(-1)
    mc = np.asarray(inputs["mean_c"], dtype=np.float64)
    mu = np.asarray(inputs["mean_u"], dtype=np.float64)
    reps = x.size // mc.size
    mc = np.tile(mc.reshape(-1), reps)
    mu = np.tile(mu.reshape(-1), reps)
    N = wl.n_steps
    M = np.empty(N, dtype=np.float64)
    MB = np.empty((N, batch), dtype=np.float64) if batch else None
    traj = [x.copy()] if keep_trajectory else None
    if wl.mode == "ddim":
        abar = (abar_cosine(wl.T) if wl.schedule == "cosine"
                else abar_linear(wl.T, wl.beta_start, wl.beta_end))
        ts = timesteps(N, wl.T, wl.spacing)
        for s in range(N):
            ab = float(abar[ts[s]])
            last = s == N - 1
            ab_prev = 1.0 if last else float(abar[ts[s + 1]])
            pc = perturb(s, "c") if perturb else None
            pu = perturb(s, "u") if perturb else None
            c = gaussian_eps(x, mc, ab, wl.data_std, pc, dt)
            u = gaussian_eps(x, mu, ab, wl.data_std, pu, dt)
            if batch:
                MB[s] = rel_mae_per_sample(c, u, batch)
            x, M[s] = ddim_step(x, c, u, dt, wv, ab, ab_prev, wl.eta, wl.seed, s, last=last)
            if keep_trajectory:
                traj.append(x.copy())
    elif wl.mode == "flow":
        t = flow_times(N)
        for s in range(N):
            c = flow_velocity(x, mc, float(t[s]), dt)
            u = flow_velocity(x, mu, float(t[s]), dt)
            if batch:
                MB[s] = rel_mae_per_sample(c, u, batch)
            x, M[s] = flow_step(x, c, u, dt, wv, float(t[s]), float(t[s + 1]))
            if keep_trajectory:
                traj.append(x.copy())
    else:
        raise ValueError(wl.mode)
    sched = schedule(M, wl.L, wl.g_slope, wl.k, wl.tau_cap)
    sched_b = ([schedule(MB[:, b], wl.L, wl.g_slope, wl.k, wl.tau_cap) for b in range(batch)]
               if batch else None)
    return RunResult(x, M, sched, traj, MB, sched_b)
