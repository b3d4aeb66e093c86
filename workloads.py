"""Seeded synthetic inputs for the CFG sampler-step workloads.

This module is the one place both sides of the parity tests take their
inputs from: the CPU oracle (``oracle/``) and the CUDA library
(``cfg_guided_sampler_step_b300``).  It holds no arithmetic of the method
(no rel-MAE, no guidance, no DDIM/Euler update, no schedule rule, no
denoiser): only the workload recipes (shapes, dtypes, sampler settings) and
seeded random draws of the starting latent, the per-branch data means of the
synthetic denoisers and the per-step perturbations.

Workloads stand in for the latents the pages run the step on:

* SD / SDXL latents (4 channels, 8x VAE downsampling; the 3840px image of the
  DistriFusion pages is a 480x480 latent),
* a 16-channel flow-matching DiT latent (the SD3 / DiT models of the xDiT
  review and of the Hybridiff notes, "Loss / training strategy": rel-MAE on
  the velocity pair),
* a 16-channel video latent (CogVideoX-style, xDiT review "long sequences").

No model weights or datasets are involved: the noise predictions come from
closed-form synthetic denoisers whose parameters are drawn here.

Random streams: every draw uses numpy's PCG64 seeded with
``SeedSequence([seed, tag(, step)])`` so each purpose has an independent,
reproducible stream:

    tag 1: x_T (the starting latent, N(0,1))
    tag 2: data mean of the conditional branch (N(0,1))
    tag 3: data mean of the unconditional branch (N(0,1))
    tag 4 / 5: per-step perturbation of the conditional / unconditional
               prediction (N(0, perturb_std^2)), keyed by the step index

Storage rounding of the drawn inputs (fp32 -> bf16, round to nearest even)
is done once here with torch's CPU cast, so both sides see the same bits.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass
from typing import Dict, Optional, Tuple

import numpy as np

TAG_XT = 1
TAG_MEAN_C = 2
TAG_MEAN_U = 3
TAG_PERTURB_C = 4
TAG_PERTURB_U = 5


@dataclass(frozen=True)
class Workload:
    """One sampler workload: latent shape, storage dtype and sampler settings.

    ``mean_shape`` is the shape of the per-branch data means; it is the latent
    shape without the batch axis (means shared across the batch) for every
    workload except the single-image point-mass one, where the means cover the
    whole latent.
    """

    name: str
    shape: Tuple[int, ...]
    dtype: str            # "f32" or "bf16" (storage); arithmetic is fp32 on the GPU
    mode: str             # "ddim" or "flow"
    n_steps: int          # denoising steps N
    w: float              # guidance scale
    eta: float            # DDIM eta (0 = deterministic); ignored for flow
    denoiser: str         # "gaussian" (std data_std; 0 = point mass) or "flow_point_mass"
    data_std: float
    perturb_std: float    # per-step N(0, perturb_std^2) added to each prediction (0 = none)
    seed: int
    T: int = 1000         # training timesteps of the linear-beta schedule
    beta_start: float = 1e-4
    beta_end: float = 0.02
    L: int = 5            # slope window of the tau1 rule
    g_slope: float = 1e-3
    k: int = 10           # tau2 = tau1 + k
    tau_cap: int = -1     # -1: global argmin of the run's own rel-MAE trace
    batch_shared_means: bool = True
    schedule: str = "linear"      # noise schedule of a DDIM workload: "linear" or "cosine"
    spacing: str = "linspace"     # DDIM timestep spacing: "linspace", "leading" or "trailing"

    @property
    def n(self) -> int:
        return int(np.prod(self.shape))

    @property
    def mean_shape(self) -> Tuple[int, ...]:
        return tuple(self.shape[1:]) if self.batch_shared_means else tuple(self.shape)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def bytes_per_step(self) -> int:
        """Algorithmic HBM bytes of one fused step: read x, pred_c, pred_u; write x."""
        return 4 * self.elem_bytes * self.n

    def scaled(self, shape: Tuple[int, ...], name: Optional[str] = None) -> "Workload":
        """The same recipe on a different latent shape (for small parity cases)."""
        return dataclasses.replace(self, shape=tuple(shape), name=name or f"{self.name}@{'x'.join(map(str, shape))}")


# The five workloads.  Parameters not stated for a workload follow the
# plainest reading: linear-beta T=1000 schedule for every DDIM workload,
# L=5, g_slope=1e-3, k=10 everywhere, data std 0.5 for every Gaussian
# denoiser, means shared across the batch.
WORKLOADS: Dict[str, Workload] = {
    "sd_point_mass_f32": Workload(
        name="sd_point_mass_f32", shape=(1, 4, 64, 64), dtype="f32", mode="ddim",
        n_steps=50, w=7.5, eta=0.0, denoiser="gaussian", data_std=0.0,
        perturb_std=0.0, seed=0, batch_shared_means=False),
    "sdxl_1024_b8_bf16": Workload(
        name="sdxl_1024_b8_bf16", shape=(8, 4, 128, 128), dtype="bf16", mode="ddim",
        n_steps=50, w=5.0, eta=0.0, denoiser="gaussian", data_std=0.5,
        perturb_std=0.0, seed=1),
    "sd_3840px_eta1_bf16": Workload(
        name="sd_3840px_eta1_bf16", shape=(1, 4, 480, 480), dtype="bf16", mode="ddim",
        n_steps=50, w=7.5, eta=1.0, denoiser="gaussian", data_std=0.5,
        perturb_std=0.05, seed=2),
    "dit_flow_b4_bf16": Workload(
        name="dit_flow_b4_bf16", shape=(4, 16, 128, 128), dtype="bf16", mode="flow",
        n_steps=28, w=3.5, eta=0.0, denoiser="flow_point_mass", data_std=0.0,
        perturb_std=0.0, seed=3),
    "video_b2_bf16": Workload(
        name="video_b2_bf16", shape=(2, 16, 13, 90, 160), dtype="bf16", mode="ddim",
        n_steps=50, w=6.0, eta=0.0, denoiser="gaussian", data_std=0.5,
        perturb_std=0.0, seed=4),
}
WORKLOAD_ORDER = list(WORKLOADS)


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest even) with torch's CPU cast; return the uint16 bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def store(a: np.ndarray, dtype: str) -> np.ndarray:
    """The stored representation of a drawn input: float32 values, or bf16 bits as uint16."""
    a32 = np.asarray(a, dtype=np.float32)
    if dtype == "f32":
        return a32.copy()
    if dtype == "bf16":
        return f32_to_bf16_bits(a32)
    raise ValueError(f"unknown storage dtype {dtype!r}")


def stored_to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact float64 values of a stored array."""
    if dtype == "f32":
        return np.asarray(a, dtype=np.float32).astype(np.float64)
    if dtype == "bf16":
        return bf16_bits_to_f32(a).astype(np.float64)
    raise ValueError(f"unknown storage dtype {dtype!r}")


def draw_inputs(wl: Workload) -> Dict[str, np.ndarray]:
    """Seeded starting latent and per-branch data means.

    Returns ``x_T`` in storage form (float32, or bf16 bits as uint16) with
    ``wl.n`` elements in C order of ``wl.shape``, and ``mean_c`` / ``mean_u``
    as float32 arrays of ``wl.mean_shape`` (exact in fp64 on both sides).
    """
    x_T = _rng(wl.seed, TAG_XT).standard_normal(wl.n)
    n_mean = int(np.prod(wl.mean_shape))
    mean_c = _rng(wl.seed, TAG_MEAN_C).standard_normal(n_mean).astype(np.float32)
    mean_u = _rng(wl.seed, TAG_MEAN_U).standard_normal(n_mean).astype(np.float32)
    return {
        "x_T": store(x_T, wl.dtype),
        "mean_c": mean_c.reshape(wl.mean_shape),
        "mean_u": mean_u.reshape(wl.mean_shape),
    }


def draw_perturbation(wl: Workload, step: int, branch: str) -> Optional[np.ndarray]:
    """Per-step N(0, perturb_std^2) perturbation of one branch's prediction (float32, n), or None."""
    if wl.perturb_std == 0.0:
        return None
    tag = TAG_PERTURB_C if branch == "c" else TAG_PERTURB_U
    p = _rng(wl.seed, tag, step).standard_normal(wl.n) * wl.perturb_std
    return p.astype(np.float32)


def draw_prediction_pair(n: int, dtype: str, seed: int, scale_c: float = 1.0,
                         scale_u: float = 1.0) -> Dict[str, np.ndarray]:
    """Independent N(0,1)-like x, pred_c, pred_u arrays for single-step tests (storage form)."""
    g = _rng(seed, 99)
    x = g.standard_normal(n)
    u = g.standard_normal(n) * scale_u
    c = u + g.standard_normal(n) * 0.1 * scale_c
    return {"x": store(x, dtype), "c": store(c, dtype), "u": store(u, dtype)}
