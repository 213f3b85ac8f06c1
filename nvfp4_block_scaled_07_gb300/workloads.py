"""Seeded synthetic workloads for the NVFP4 MoE expert layer.

This module only draws random inputs; it holds none of the layer's
arithmetic (no quantisation, routing or GEMM), so both the CUDA path and the
CPU oracle can take their inputs from it.

The five layer shapes follow the workloads the source pages measure: the
GLM-5-NVFP4 decode regime with 256 experts and about 16-64 rows per expert
("Uncovering SM120 CUTLASS Collective Implementations", Context;
"Discovering SM120-Specific CUTLASS MoE Kernels", Assumptions: E=256), plus a
tiny case, a skewed-routing case and a prefill-sized case.  No dataset or
trained weight is involved: logits and activations are N(0, 1), weights are
N(0, 0.02), all drawn in float32 and rounded to bfloat16 where the layer
takes bfloat16.

Two generators exist:
  * ``host_inputs``   numpy ``default_rng(seed)``, fixed draw order
                      (logits, x, W_gu, W_d); used where the oracle runs on
                      every token.
  * ``device_inputs`` ``torch.Generator`` on the GPU with the same seed and
                      draw order; used for full-size shapes (tens of GB of
                      weights), where the oracle checks sampled outputs
                      copied back to the host.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int              # tokens
    E: int              # experts
    k: int              # experts per token
    H: int              # hidden size (K of gate/up, N of down)
    I: int              # expert intermediate size (K of down)
    score: str          # "softmax" or "sigmoid"
    renormalize: bool = True
    zipf_s: float = 0.0  # > 0: add a Zipf(s) popularity bias to the logits
    w_std: float = 0.02
    h_scale: float = 2.0 ** -4   # static per-tensor scale of the SwiGLU output

    @property
    def R(self):
        return self.T * self.k

    def describe(self):
        d = dataclasses.asdict(self)
        return {k: v for k, v in d.items() if k != "name"}


WORKLOADS = {
    "tiny": Workload("tiny", T=16, E=8, k=2, H=256, I=128, score="softmax"),
    "decode_t128": Workload("decode_t128", T=128, E=256, k=8, H=6144, I=2048, score="sigmoid"),
    "decode_t1024": Workload("decode_t1024", T=1024, E=256, k=8, H=6144, I=2048, score="sigmoid"),
    "skewed_t2048": Workload("skewed_t2048", T=2048, E=256, k=8, H=6144, I=2048, score="sigmoid",
                             zipf_s=1.1),
    "prefill_t16384": Workload("prefill_t16384", T=16384, E=64, k=8, H=7168, I=4096, score="sigmoid"),
}

# A small decode-regime layer for profiler captures: the decode shape with
# 16 experts (~4 rows each, 340 MB of NVFP4 weights: larger than L2, small
# enough for multi-pass counter collection).
PROFILE_WORKLOADS = {
    "profile_decode_e16": Workload("profile_decode_e16", T=8, E=16, k=8, H=6144, I=2048, score="sigmoid"),
    "profile_prefill_e8": Workload("profile_prefill_e8", T=2048, E=8, k=8, H=7168, I=4096, score="sigmoid"),
    # the skewed_t2048 regime (Zipf 1.1 popularity: a few hot experts with hundreds of rows next to
    # many cold ones with a handful) at a quarter of the experts and tokens: 1.4 GB of NVFP4 weights
    "profile_skewed_e64": Workload("profile_skewed_e64", T=512, E=64, k=8, H=6144, I=2048, score="sigmoid",
                                   zipf_s=1.1),
    # the prepare kernel's work of skewed_t2048 and prefill_t16384 (the same T, E, k, H and routing)
    # with I = 128, so the weights are small and a multi-pass capture of the prepare holds little memory
    "profile_prepare_t2048": Workload("profile_prepare_t2048", T=2048, E=256, k=8, H=6144, I=128,
                                      score="sigmoid", zipf_s=1.1),
    "profile_prepare_t16384": Workload("profile_prepare_t16384", T=16384, E=64, k=8, H=7168, I=128,
                                       score="sigmoid"),
}

# Medium shapes that the oracle finishes in seconds but that still span
# several tiles per expert, ragged expert sizes and a partial K tile.
TEST_WORKLOADS = {
    "ragged_small": Workload("ragged_small", T=96, E=8, k=2, H=512, I=384, score="sigmoid"),
    "many_experts": Workload("many_experts", T=64, E=32, k=4, H=384, I=256, score="sigmoid"),
    "wide_experts": Workload("wide_experts", T=300, E=4, k=2, H=1024, I=256, score="softmax"),
    "zipf_small": Workload("zipf_small", T=256, E=16, k=4, H=384, I=128, score="sigmoid", zipf_s=1.1),
}


def zipf_bias(E, s):
    """Per-expert logit bias -s * ln(e + 1): expert e has Zipf(s) popularity rank e+1."""
    return (-s * np.log(np.arange(1, E + 1, dtype=np.float64))).astype(np.float32)


def _to_bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def host_inputs(w: Workload, seed: int = 0, with_weights: bool = True):
    """CPU tensors: logits f32 [T,E], bias f32 [E] or None, x bf16 [T,H],
    w_gu bf16 [E,2I,H] (gate rows first), w_d bf16 [E,H,I]."""
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((w.T, w.E), dtype=np.float32)
    x = _to_bf16(rng.standard_normal((w.T, w.H), dtype=np.float32))
    out = dict(logits=torch.from_numpy(logits),
               bias=torch.from_numpy(zipf_bias(w.E, w.zipf_s)) if w.zipf_s > 0 else None,
               x=x)
    if with_weights:
        out["w_gu"] = _to_bf16(rng.standard_normal((w.E, 2 * w.I, w.H), dtype=np.float32) * np.float32(w.w_std))
        out["w_d"] = _to_bf16(rng.standard_normal((w.E, w.H, w.I), dtype=np.float32) * np.float32(w.w_std))
    return out


def device_inputs(w: Workload, seed: int = 0, device="cuda", with_weights: bool = True):
    """Same tensors as host_inputs, drawn on the device with torch.Generator.

    Weights are drawn one expert at a time so the float32 temporaries stay
    small; the result is bf16.
    """
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    logits = torch.randn((w.T, w.E), generator=g, device=device, dtype=torch.float32)
    x = torch.randn((w.T, w.H), generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    out = dict(logits=logits,
               bias=torch.from_numpy(zipf_bias(w.E, w.zipf_s)).to(device) if w.zipf_s > 0 else None,
               x=x)
    if with_weights:
        w_gu = torch.empty((w.E, 2 * w.I, w.H), device=device, dtype=torch.bfloat16)
        w_d = torch.empty((w.E, w.H, w.I), device=device, dtype=torch.bfloat16)
        for e in range(w.E):
            w_gu[e] = (torch.randn((2 * w.I, w.H), generator=g, device=device) * w.w_std).to(torch.bfloat16)
        for e in range(w.E):
            w_d[e] = (torch.randn((w.H, w.I), generator=g, device=device) * w.w_std).to(torch.bfloat16)
        out["w_gu"], out["w_d"] = w_gu, w_d
    return out


def random_nvfp4_operand(rows, K, seed, scale_lo=0x20, scale_hi=0x48):
    """Random NVFP4 operand bytes for GEMM-only tests: uniformly random packed
    codes [rows, K/2], scale bytes uniform in [scale_lo, scale_hi] (row-major
    [rows, K/16]) and a per-tensor scale.  Pure random bytes, no quantiser."""
    rng = np.random.default_rng(seed)
    packed = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    scales = rng.integers(scale_lo, scale_hi + 1, size=(rows, K // 16), dtype=np.uint8)
    s = np.float32(rng.uniform(0.01, 0.1))
    return packed, scales, s


def random_routing(T, E, k, seed, counts_hint=None):
    """Random top-k expert ids [T,k] (distinct per token) for permute tests."""
    rng = np.random.default_rng(seed)
    if counts_hint is None:
        return np.stack([rng.choice(E, size=k, replace=False) for _ in range(T)]).astype(np.int32)
    p = np.asarray(counts_hint, dtype=np.float64)
    p = p / p.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)


def algorithmic_flops(w: Workload):
    """6*T*k*H*I: gate/up 4*R*H*I plus down 2*R*I*H, routed rows only."""
    return 6.0 * w.T * w.k * w.H * w.I


def nvfp4_bytes(n_elems):
    """Bytes of n NVFP4 elements with their scales: 0.5 + 1/16 per element."""
    return n_elems * (0.5 + 1.0 / 16.0)


def mxfp4_bytes(n_elems):
    """Bytes of n MXFP4 elements with their scales: 0.5 + 1/32 per element."""
    return n_elems * (0.5 + 1.0 / 32.0)


def fp4_bytes(n_elems, fmt="nvfp4"):
    return mxfp4_bytes(n_elems) if fmt == "mxfp4" else nvfp4_bytes(n_elems)


def ceil_div(a, b):
    return -(-a // b)


__all__ = ["Workload", "WORKLOADS", "PROFILE_WORKLOADS", "TEST_WORKLOADS", "host_inputs", "device_inputs",
           "random_nvfp4_operand", "random_routing", "zipf_bias", "algorithmic_flops",
           "nvfp4_bytes", "ceil_div"]
