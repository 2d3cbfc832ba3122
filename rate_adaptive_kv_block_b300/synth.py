"""Seeded synthetic K/V inputs.

This module only draws random tensors: it holds none of the quantizer's
arithmetic, and both the CUDA path's tests/benchmark and the CPU oracle's
tests take their inputs from it.

Distributions (per workload):
  * "scaled normal": N(0,1) entries times a per-(stream, channel) scale
    exp(N(0, 0.5^2)) (log-normal with log-std 0.5);
  * "scaled normal + outliers": as above, with 4 channels (the first 4 of one
    seeded permutation of the D channels, the same for every stream) x10;
  * "student-t(5)": Z / sqrt(chi2_5 / 5), chi2_5 a sum of 5 squared normals;
  * "hadamard-rotated normal": N(0,1) rows times H_D / sqrt(D), H_D the
    Sylvester-order Hadamard matrix.
Every draw is rounded to binary16 (round to nearest even).

Two backends: numpy (CPU, PCG64 from numpy.random.default_rng) and torch
(CUDA Philox from torch.Generator) for the multi-GB workloads.  The two give
different numbers for the same seed; each is deterministic for its seed.
"""
from dataclasses import dataclass, field
from typing import List, Optional, Tuple

import numpy as np


@dataclass
class Workload:
    name: str
    S: int                  # streams (layer x K/V x head [x sequence])
    T: int                  # tokens per stream (multiple of 32)
    D: int                  # head dim
    G: int                  # features per block (D, or a feature group)
    s: int                  # max levels per block
    budgets: List[float]    # bits per entry
    parts: List[Tuple[str, int]] = field(default_factory=list)  # (dist, streams)
    eta: Optional[float] = None     # subgradient step (decode admission)

    @property
    def entries(self) -> int:
        return self.S * self.T * self.D

    @property
    def nblocks(self) -> int:
        return self.S * (self.T // 32) * (self.D // self.G)


def workload(name: str, T: Optional[int] = None, S: Optional[int] = None) -> Workload:
    """The five synthetic workloads; T / S override the sizes (for tests that
    need the same distribution at a size a CPU check finishes quickly)."""
    if name == "k_head_small":
        w = Workload(name, 8, 256, 128, 128, 8, [3.0], [("scaled_normal", 8)])
    elif name == "llama3_8b_layer":
        w = Workload(name, 16, 8192, 128, 128, 16, [2.5],
                     [("scaled_normal_outliers", 8), ("student_t5", 8)])
    elif name == "full_model_cache":
        w = Workload(name, 512, 32768, 128, 128, 16, [2.0],
                     [("scaled_normal", 512)])
    elif name == "decode_admission":
        w = Workload(name, 32768, 32, 128, 128, 16, [2.5],
                     [("scaled_normal", 32768)], eta=1e-6)
    elif name == "hadamard_groups":
        w = Workload(name, 8, 131072, 128, 32, 16, [1.5, 2.0, 3.0, 4.0],
                     [("hadamard_normal", 8)])
    else:
        raise KeyError(name)
    if T is not None:
        w.T = T
    if S is not None:
        # keep the same mix of distributions, scaled to the new stream count
        tot = sum(n for _, n in w.parts)
        parts = [(d, max(1, n * S // tot)) for d, n in w.parts]
        parts[-1] = (parts[-1][0], S - sum(n for _, n in parts[:-1]))
        w.parts = parts
        w.S = S
    return w


WORKLOADS = ["k_head_small", "llama3_8b_layer", "full_model_cache",
             "decode_admission", "hadamard_groups"]


def hadamard(n: int) -> np.ndarray:
    """Sylvester-order Hadamard matrix H_n (n a power of two), entries +-1."""
    H = np.ones((1, 1), dtype=np.float32)
    while H.shape[0] < n:
        H = np.block([[H, H], [H, -H]])
    return H


def _np_part(dist: str, S: int, T: int, D: int, rng) -> np.ndarray:
    if dist in ("scaled_normal", "scaled_normal_outliers"):
        z = rng.standard_normal((S, T, D), dtype=np.float32)
        scale = np.exp(0.5 * rng.standard_normal((S, 1, D), dtype=np.float32))
        if dist == "scaled_normal_outliers":
            ch = rng.permutation(D)[:4]
            scale[:, :, ch] *= 10.0
        return z * scale
    if dist == "student_t5":
        z = rng.standard_normal((S, T, D), dtype=np.float32)
        chi2 = np.zeros((S, T, D), dtype=np.float32)
        for _ in range(5):
            chi2 += rng.standard_normal((S, T, D), dtype=np.float32) ** 2
        return z / np.sqrt(chi2 / 5.0)
    if dist == "hadamard_normal":
        z = rng.standard_normal((S, T, D), dtype=np.float32)
        H = hadamard(D) / np.float32(np.sqrt(D))
        return z @ H
    raise KeyError(dist)


def make_numpy(w: Workload, seed: int = 0) -> np.ndarray:
    """[S, T, D] uint16 array of binary16 bit patterns (CPU backend)."""
    rng = np.random.default_rng(seed)
    out = [_np_part(d, n, w.T, w.D, rng) for d, n in w.parts]
    x = np.concatenate(out, axis=0).astype(np.float16)
    return x.view(np.uint16)


def make_torch(w: Workload, seed: int = 0, device: str = "cuda"):
    """[S, T, D] torch.float16 tensor on `device` (torch backend).  Generated
    in chunks of streams so the fp32 temporaries stay small."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.empty((w.S, w.T, w.D), dtype=torch.float16, device=device)
    row = 0
    chunk = max(1, (1 << 26) // (w.T * w.D))
    H = None
    for dist, n in w.parts:
        ch = None
        if dist == "scaled_normal_outliers":
            ch = torch.randperm(w.D, generator=g, device=device)[:4]
        for s0 in range(0, n, chunk):
            m = min(chunk, n - s0)
            shp = (m, w.T, w.D)
            if dist in ("scaled_normal", "scaled_normal_outliers"):
                z = torch.randn(shp, generator=g, device=device)
                sc = torch.exp(0.5 * torch.randn((m, 1, w.D), generator=g,
                                                 device=device))
                if ch is not None:
                    sc[:, :, ch] *= 10.0
                v = z * sc
            elif dist == "student_t5":
                z = torch.randn(shp, generator=g, device=device)
                c2 = torch.zeros(shp, device=device)
                for _ in range(5):
                    c2 += torch.randn(shp, generator=g, device=device) ** 2
                v = z / torch.sqrt(c2 / 5.0)
            elif dist == "hadamard_normal":
                if H is None:
                    H = torch.from_numpy(hadamard(w.D) / np.float32(np.sqrt(w.D))).to(device)
                v = torch.randn(shp, generator=g, device=device) @ H
            else:
                raise KeyError(dist)
            x[row:row + m] = v.to(torch.float16)
            row += m
    return x


# ------------------------------------------------ distortion weights
# Seeded per-entry weights with the structure of attention sensitivity
# measured on a calibration batch: the first ceil(S/2) streams are keys, whose
# error reaches the logits through q . dk, so their weight depends on the
# feature only (the mean squared query component: log-normal with log-std 1,
# and 4 outlier channels x25); the other streams are values, whose error
# reaches the output through sum_t p_t dv_t, so their weight depends on the
# token only (the mean squared attention probability: log-normal with log-std
# 1.5, and the first 4 tokens, attention sinks, x50).  Each stream's weights
# are scaled to mean 1.  Random draws only; float32 [S, T, D].

def _key_weights_np(n, D, rng):
    w = np.exp(rng.standard_normal((n, 1, D), dtype=np.float32))
    w[:, :, rng.permutation(D)[:4]] *= 25.0
    return w / w.mean(axis=2, keepdims=True)


def _value_weights_np(n, T, rng):
    w = np.exp(1.5 * rng.standard_normal((n, T, 1), dtype=np.float32))
    w[:, :4, :] *= 50.0
    return w / w.mean(axis=1, keepdims=True)


def weights_numpy(w: Workload, seed: int = 0) -> np.ndarray:
    """[S, T, D] float32 distortion weights (CPU backend)."""
    rng = np.random.default_rng(seed)
    nk = (w.S + 1) // 2
    out = np.empty((w.S, w.T, w.D), dtype=np.float32)
    out[:nk] = _key_weights_np(nk, w.D, rng)
    out[nk:] = _value_weights_np(w.S - nk, w.T, rng)
    return out


def weights_torch(w: Workload, seed: int = 0, device: str = "cuda"):
    """[S, T, D] float32 distortion weights on `device` (torch backend)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    nk = (w.S + 1) // 2
    out = torch.empty((w.S, w.T, w.D), dtype=torch.float32, device=device)
    kw = torch.exp(torch.randn((nk, 1, w.D), generator=g, device=device))
    kw[:, :, torch.randperm(w.D, generator=g, device=device)[:4]] *= 25.0
    out[:nk] = kw / kw.mean(dim=2, keepdim=True)
    vw = torch.exp(1.5 * torch.randn((w.S - nk, w.T, 1), generator=g, device=device))
    vw[:, :4, :] *= 50.0
    out[nk:] = vw / vw.mean(dim=1, keepdim=True)
    return out
