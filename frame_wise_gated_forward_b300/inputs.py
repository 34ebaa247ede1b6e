"""Seeded synthetic inputs for the frame-wise GDN forward.

This module holds no arithmetic of the method itself: it only draws random
tensors with the distributions of the workloads and rounds them to the dtypes
the C ABI takes.  Both the CUDA path and the CPU oracle are fed from here.

Workload shapes come from the SANA-WM pages: a 60 s, 16 fps, 720p clip
(article "NVIDIA's New 2.6B World Model...", intro and "The Architecture")
with 8 raw frames per latent frame ("Camera Control") and native 8k+1 windows
(WorldFoundry model card, "What it is for") gives F = 8*15 + 1 = 121 latent
frames; a 1280x704 frame (model card intro) at 32x spatial compression gives a
40x22 grid, N = 880 tokens per frame.

Distributions (one CPU ``torch.Generator`` per stream, seeded; the draw order
is fixed as q, k, v, beta, alpha, S_0):
  q, k  ~ N(0, 1), L2-normalised per (token, head) in fp32, then rounded to
          bf16 with round-to-nearest-even;
  v     ~ N(0, 1), rounded to bf16;
  beta  = sigmoid(N(0, 1)) / N                      fp32 [B, F, N, H]
  alpha = exp(-softplus(N(0, 1)) * 0.05)            fp32 [B, F, H]  (no clamp)
  S_0   = 0, or N(0, 0.01) read as variance 0.01 (std 0.1), fp32 [B, H, dv, dk]
For the 8-bit entry points (draw_fp8) q, k and v are instead quantized to
OCP FP8 E4M3 with one fp32 scale per tensor (amax / 448, round to nearest
even).
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    F: int
    N: int
    dk: int
    dv: int
    # per batch stream: (seed, S_0 std or 0.0)
    streams: tuple
    # True: F sequential single-frame step calls, frame f drawn from seed+f
    streaming: bool = False

    @property
    def tokens(self) -> int:
        return self.B * self.F * self.N


WORKLOADS = {
    # tiny case the oracle finishes instantly; fp32 draws through the bf16 ABI
    "tiny": Workload("tiny", 1, 2, 4, 16, 32, 32, ((0, 0.0),)),
    # one 9-latent-frame native window (8k+1, k=1) at 1280x704
    "window9": Workload("window9", 1, 8, 9, 880, 64, 64, ((0, 0.1),)),
    # the 60 s 720p sequence: 121 x 880 = 106,480 tokens, 16 heads, d = 128
    "seq60s": Workload("seq60s", 1, 16, 121, 880, 128, 128, ((0, 0.0),)),
    # guidance-doubled batch: two independent streams, second with S_0 != 0
    "cfg2": Workload("cfg2", 2, 16, 121, 880, 128, 128, ((0, 0.0), (1, 0.1))),
    # interactive rollout: 121 single-frame steps on a resident state
    "stream121": Workload("stream121", 1, 16, 121, 880, 128, 128, ((0, 0.0),),
                          streaming=True),
}


def _draw_f32(B, H, F, N, dk, dv, seed, s0_std):
    """The fp32 draws shared by draw() and draw_fp8(): q, k L2-normalised."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((B, F, N, H, dk), generator=g, dtype=torch.float32)
    k = torch.randn((B, F, N, H, dk), generator=g, dtype=torch.float32)
    v = torch.randn((B, F, N, H, dv), generator=g, dtype=torch.float32)
    braw = torch.randn((B, F, N, H), generator=g, dtype=torch.float32)
    araw = torch.randn((B, F, H), generator=g, dtype=torch.float32)
    if s0_std > 0.0:
        s0 = torch.randn((B, H, dv, dk), generator=g, dtype=torch.float32) * s0_std
    else:
        s0 = torch.zeros((B, H, dv, dk), dtype=torch.float32)
    q = torch.nn.functional.normalize(q, dim=-1)
    k = torch.nn.functional.normalize(k, dim=-1)
    beta = torch.sigmoid(braw) / float(max(N, 1))
    alpha = torch.exp(-torch.nn.functional.softplus(araw) * 0.05)
    return q, k, v, alpha.contiguous(), beta.contiguous(), s0.contiguous()


def draw(B: int, H: int, F: int, N: int, dk: int, dv: int, seed: int,
         s0_std: float = 0.0) -> dict:
    """Draw one set of inputs (all batch rows from one generator)."""
    q, k, v, alpha, beta, s0 = _draw_f32(B, H, F, N, dk, dv, seed, s0_std)
    return {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16),
            "alpha": alpha, "beta": beta, "state_in": s0}


E4M3_MAX = 448.0


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor scaled OCP FP8 E4M3: scale = amax / 448 (fp32), codes =
    round-to-nearest-even(x / scale) as torch.float8_e4m3fn, returned as
    their uint8 bytes.  Input preparation only: the method itself never
    quantizes."""
    amax = float(x.abs().max())
    scale = amax / E4M3_MAX if amax > 0.0 else 1.0
    codes = (x / scale).to(torch.float8_e4m3fn).view(torch.uint8).contiguous()
    return codes, float(scale)


def draw_fp8(B: int, H: int, F: int, N: int, dk: int, dv: int, seed: int,
             s0_std: float = 0.0) -> dict:
    """The draws of draw() with q, k and v quantized to per-tensor-scaled
    e4m3 instead of rounded to bf16 (same generator sequence)."""
    q, k, v, alpha, beta, s0 = _draw_f32(B, H, F, N, dk, dv, seed, s0_std)
    q8, sq = quantize_e4m3(q)
    k8, sk = quantize_e4m3(k)
    v8, sv = quantize_e4m3(v)
    return {"q8": q8, "k8": k8, "v8": v8, "q_scale": sq, "k_scale": sk, "v_scale": sv,
            "alpha": alpha, "beta": beta, "state_in": s0}


E2M1_MAX = 6.0
# the eight non-negative E2M1 magnitudes, in code order (codes 0..7)
E2M1_MAGNITUDES = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def quantize_nvfp4(x: torch.Tensor):
    """NVFP4 with 16-element blocks along the last dimension: one fp32 tensor
    scale gs = amax / (6 * 448), one E4M3 block scale per 16 elements
    (round-to-nearest-even of block amax / (6 gs)), and E2M1 codes, each the
    nearest E2M1 value to x / (gs * block scale) (ties to the even code).
    Returns (packed uint8 [..., d/2] with element 2i in the low nibble, block
    scale codes uint8 [..., d/16], gs).  Input preparation only: the method
    itself never quantizes."""
    d = x.shape[-1]
    if d % 16:
        raise ValueError("the last dimension must be a multiple of 16")
    x = x.to(torch.float32)
    amax = float(x.abs().max())
    gs = amax / (E2M1_MAX * E4M3_MAX) if amax > 0.0 else 1.0
    xb = x.reshape(*x.shape[:-1], d // 16, 16)
    sc = (xb.abs().amax(dim=-1) / (E2M1_MAX * gs)).to(torch.float8_e4m3fn)
    den = (sc.to(torch.float32) * gs).unsqueeze(-1)
    y = torch.where(den > 0, xb / torch.where(den > 0, den, torch.ones_like(den)), torch.zeros_like(xb))
    mags = torch.tensor(E2M1_MAGNITUDES, dtype=torch.float32)
    a = y.abs().clamp(max=E2M1_MAX)
    dist = (a.unsqueeze(-1) - mags).abs()                 # [..., 16, 8]
    best = dist.min(dim=-1, keepdim=True).values
    idx = torch.arange(8)
    # among the nearest magnitudes, the even code (mantissa bit 0) wins a tie
    key = torch.where(dist == best, (idx % 2) * 8 + idx, torch.full_like(idx, 99))
    code = key.argmin(dim=-1).to(torch.uint8)
    code = code | ((y < 0).to(torch.uint8) << 3)
    code = code.reshape(*x.shape[:-1], d)
    packed = (code[..., 0::2] | (code[..., 1::2] << 4)).contiguous()
    return packed, sc.view(torch.uint8).contiguous(), float(gs)


def draw_nvfp4(B: int, H: int, F: int, N: int, dk: int, dv: int, seed: int,
               s0_std: float = 0.0) -> dict:
    """The draws of draw() with q, k and v quantized to NVFP4 (same generator
    sequence)."""
    q, k, v, alpha, beta, s0 = _draw_f32(B, H, F, N, dk, dv, seed, s0_std)
    out = {"alpha": alpha, "beta": beta, "state_in": s0}
    for name, t in (("q", q), ("k", k), ("v", v)):
        out[name + "4"], out[name + "_sf"], out[name + "_gs"] = quantize_nvfp4(t)
    return out


def workload_inputs(w: Workload) -> dict:
    """Inputs of a named workload, concatenated over its batch streams.

    For a streaming workload frame f is drawn from seed (stream seed + f) as a
    one-frame draw; the frames are concatenated along F, and the initial
    state is that of the stream (zero for the shipped workload).
    """
    parts = []
    for seed, std in w.streams:
        if w.streaming:
            frames = [draw(1, w.H, 1, w.N, w.dk, w.dv, seed + f, 0.0) for f in range(w.F)]
            p = {name: torch.cat([fr[name] for fr in frames], dim=1)
                 for name in ("q", "k", "v", "alpha", "beta")}
            if std > 0.0:
                p["state_in"] = draw(1, w.H, 1, 1, w.dk, w.dv, seed, std)["state_in"]
            else:
                p["state_in"] = torch.zeros((1, w.H, w.dv, w.dk), dtype=torch.float32)
            parts.append(p)
        else:
            parts.append(draw(1, w.H, w.F, w.N, w.dk, w.dv, seed, std))
    return {name: torch.cat([p[name] for p in parts], dim=0).contiguous()
            for name in parts[0]}


def has_zero_state(w: Workload) -> bool:
    return all(std == 0.0 for _, std in w.streams)


def draw_raw(B: int, H: int, F: int, N: int, dk: int, dv: int, seed: int,
             qk_std: float = 1.0, s0_std: float = 0.0) -> dict:
    """Raw inputs for the folded-prologue entry points: unnormalized q, k
    ~ N(0, qk_std^2) (bf16), v ~ N(0, 1) (bf16), decay logits a ~ N(0, 1)
    [B, F, H] and write-strength logits b ~ N(0, 1) - ln N [B, F, N, H], so that
    sigmoid(b) is about 1/N per token, as in the normalized workloads."""
    import math
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = (torch.randn((B, F, N, H, dk), generator=g) * qk_std).to(torch.bfloat16)
    k = (torch.randn((B, F, N, H, dk), generator=g) * qk_std).to(torch.bfloat16)
    v = torch.randn((B, F, N, H, dv), generator=g).to(torch.bfloat16)
    b = torch.randn((B, F, N, H), generator=g) - math.log(max(N, 1))
    a = torch.randn((B, F, H), generator=g)
    if s0_std > 0.0:
        s0 = torch.randn((B, H, dv, dk), generator=g) * s0_std
    else:
        s0 = torch.zeros((B, H, dv, dk))
    return {"q": q, "k": k, "v": v, "a_logit": a.contiguous(), "b_logit": b.contiguous(),
            "state_in": s0.contiguous()}


def draw_delta(B: int, H: int, F: int, N: int, dk: int, dv: int, seed: int,
               s0_std: float = 0.0, keys: str = "shared", mass=(0.5, 0.95),
               noise: float = 0.3) -> dict:
    """Inputs in the regime where the delta-rule correction dominates the
    update (SANA-WM article, "The Architecture": the state is corrected by a
    delta rule, not only accumulated): |K_f^T B_f K_f| is close to 1 in every
    frame, so S (I - A_f) differs from S by a large term instead of the ~0.4 %
    of the spec's beta = sigmoid(x)/N workloads.

    keys = "shared": per (b, f, h) one unit direction u; token keys
        k_n = normalize(u + noise * g_n / sqrt(dk)), g_n ~ N(0, I), so the
        keys of a frame are strongly correlated; beta_n = m * w_n / sum(w)
        with w_n = sigmoid(N(0, 1)) and m ~ U(mass) per (b, f, h), i.e.
        sum_n beta_n |k_n|^2 = m before the bf16 rounding of k.
    keys = "orthonormal" (needs N <= dk): the keys of a frame are the first N
        rows of a random orthogonal matrix and beta_n ~ U(0.5, 1), so A_f has
        eigenvalues beta_n up to 1 (a near-projection: exact delta writes).
    q ~ N(0, 1) L2-normalised, v ~ N(0, 1), alpha as in draw(); q, k, v rounded
    to bf16.  Input preparation only: no arithmetic of the method."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.nn.functional.normalize(torch.randn((B, F, N, H, dk), generator=g), dim=-1)
    v = torch.randn((B, F, N, H, dv), generator=g)
    araw = torch.randn((B, F, H), generator=g)
    alpha = torch.exp(-torch.nn.functional.softplus(araw) * 0.05)
    if keys == "shared":
        u = torch.nn.functional.normalize(torch.randn((B, F, 1, H, dk), generator=g), dim=-1)
        gk = torch.randn((B, F, N, H, dk), generator=g)
        k = torch.nn.functional.normalize(u + noise * gk / float(dk) ** 0.5, dim=-1)
        w = torch.sigmoid(torch.randn((B, F, N, H), generator=g))
        m = mass[0] + (mass[1] - mass[0]) * torch.rand((B, F, 1, H), generator=g)
        beta = m * w / w.sum(dim=2, keepdim=True)
    elif keys == "orthonormal":
        if N > dk:
            raise ValueError("orthonormal keys need N <= dk")
        z = torch.randn((B, F, H, dk, dk), generator=g, dtype=torch.float64)
        qm, _ = torch.linalg.qr(z)                          # columns orthonormal
        k = qm.transpose(-1, -2)[..., :N, :].permute(0, 1, 3, 2, 4).to(torch.float32)   # [B, F, N, H, dk]
        beta = 0.5 + 0.5 * torch.rand((B, F, N, H), generator=g)
    else:
        raise ValueError(f"unknown key mode {keys!r}")
    if s0_std > 0.0:
        s0 = torch.randn((B, H, dv, dk), generator=g) * s0_std
    else:
        s0 = torch.zeros((B, H, dv, dk))
    return {"q": q.to(torch.bfloat16).contiguous(), "k": k.to(torch.bfloat16).contiguous(),
            "v": v.to(torch.bfloat16).contiguous(), "alpha": alpha.contiguous(),
            "beta": beta.to(torch.float32).contiguous(), "state_in": s0.contiguous()}
