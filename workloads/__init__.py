"""Seeded synthetic inputs for the SDM forward step.

This module holds the workload shapes and the random-number recipe that both
the CUDA path and the oracle consume.  It holds none of the method's
arithmetic: it only draws tensors.

Recipe (one ``torch.Generator('cpu')`` seeded with the workload's seed, draws
in this order): q_w, q_r ~ N(0,1)*qk_std; K ~ N(0,1)*qk_std; v ~ N(0,1);
alpha ~ U(0.9, 1); beta ~ U(0, 1); M_0 ~ N(0,1)*0.02.  Draws are float32; the
tensors that a workload marks bf16 (q_w, q_r, K, v, alpha, beta) are rounded to
bf16 once, and both sides read those same rounded values.  M_0 is always fp32.

Tables too large to draw on the host (the decode workloads' tens of GB) are
drawn with the same recipe by a generator on the device (``device=`` below):
the same distributions and order, different numbers; only timing runs use it.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    n_sub: int
    d_h: int
    d_v: int
    W: int
    R: int
    bf16: bool          # q, K, v, alpha, beta stored as bf16 (state stays fp32)
    score_kind: int     # 0 dot product, 1 inverse distance
    qk_std: float
    seed: int
    k_w: int = 0
    k_r: int = 0
    idw_eps: float = 1e-3
    update_form: int = 0

    @property
    def N(self) -> int:
        return self.n_sub * self.n_sub

    @property
    def tokens(self) -> int:
        return self.B * self.T

    @property
    def token_heads(self) -> int:
        return self.B * self.H * self.T

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads: a tiny fp32 case, a mid-size bf16 case, the GDN-matched
# scale (N = 65536 slots, W = R = 64, d_v = 128), an FwPKM-shaped table with
# inverse-distance scores, and a long single-sequence scan.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 256, 32, 16, 32, 8, 8, False, 0, 0.25, 0),
    "mid": Workload("mid", 4, 4, 2048, 128, 64, 128, 64, 64, True, 0, 0.25, 1),
    "gdn_matched": Workload("gdn_matched", 8, 8, 4096, 256, 64, 128, 64, 64, True, 0, 0.25, 2),
    "fwpkm_idw": Workload("fwpkm_idw", 4, 1, 8192, 512, 256, 512, 8, 8, False, 1, 1.0, 3),
    "long_seq": Workload("long_seq", 1, 16, 131072, 256, 64, 128, 64, 64, True, 0, 0.25, 4),
    # Decode (one token per sequence and call) at the per-head shapes of the
    # 1.4B (sqrt N = 240, d_v = 960) and 8B (sqrt N = 480, d_v = 1920) models,
    # two heads each.
    "decode_l08": Workload("decode_l08", 64, 2, 1, 240, 64, 960, 64, 64, True, 0, 0.25, 5),
    "decode_l13": Workload("decode_l13", 16, 2, 1, 480, 64, 1920, 64, 64, True, 0, 0.25, 6),
}
ORDER = ["tiny", "mid", "gdn_matched", "fwpkm_idw", "long_seq"]


def generate(w: Workload, dtype_override=None, device=None):
    """Draw the inputs of workload ``w`` (on the CPU unless ``device``).

    Returns a dict of tensors: q_w, q_r [B,H,T,2,d_h]; K [H,2,s,d_h];
    v [B,H,T,d_v]; alpha, beta [B,H,T] (bf16 or fp32); M0 [B,H,N,d_v] fp32.
    """
    dev = torch.device(device or "cpu")
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    B, H, T, s, dh, dv = w.B, w.H, w.T, w.n_sub, w.d_h, w.d_v
    kw = dict(generator=g, device=dev)
    q_w = torch.randn(B, H, T, 2, dh, **kw) * w.qk_std
    q_r = torch.randn(B, H, T, 2, dh, **kw) * w.qk_std
    K = torch.randn(H, 2, s, dh, **kw) * w.qk_std
    v = torch.randn(B, H, T, dv, **kw)
    alpha = torch.rand(B, H, T, **kw) * 0.1 + 0.9
    beta = torch.rand(B, H, T, **kw)
    M0 = torch.randn(B, H, s * s, dv, **kw) * 0.02
    dt = dtype_override or (torch.bfloat16 if w.bf16 else torch.float32)
    out = dict(q_w=q_w, q_r=q_r, K=K, v=v, alpha=alpha, beta=beta)
    out = {k: t.to(dt).contiguous() for k, t in out.items()}
    out["M0"] = M0.contiguous()
    return out


def chain_slice(inputs: dict, b: int, h: int) -> dict:
    """Inputs of one (b, h) chain as B=1, H=1 tensors (K keeps head h only)."""
    return dict(
        q_w=inputs["q_w"][b:b + 1, h:h + 1].contiguous(),
        q_r=inputs["q_r"][b:b + 1, h:h + 1].contiguous(),
        K=inputs["K"][h:h + 1].contiguous(),
        v=inputs["v"][b:b + 1, h:h + 1].contiguous(),
        alpha=inputs["alpha"][b:b + 1, h:h + 1].contiguous(),
        beta=inputs["beta"][b:b + 1, h:h + 1].contiguous(),
        M0=inputs["M0"][b:b + 1, h:h + 1].contiguous(),
    )
