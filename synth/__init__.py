"""Seeded synthetic inputs for the routed-MoE expert layer.

This module only *makes data*: router logits, bf16 activations and expert
weights already encoded in the storage formats the layer consumes (MXFP4 codes
+ E8M0 scales, and the Q2_K-style 2-bit super-blocks).  Both the CUDA path and
the CPU oracle receive the bytes produced here; neither side's arithmetic lives
in this file (the layer only ever *decodes* these formats, never encodes them).

Workloads (the pages give no layer shapes; the shapes below are the layer
specification this library is built for):

=========  ====  =====  ===  ====  =  ==========================================
name       T     d      E    f     k  routing recipe
=========  ====  =====  ===  ====  =  ==========================================
tiny       4     256    8    128   2  randperm(0..7)*0.5 + N(0, 0.01)
decode1    1     4096   256  2048  8  N(0,1), tie-free jitter
decode64   64    4096   256  2048  8  N(0,1) + log Zipf(1.1) prior (global)
prefill    4096  4096   256  2048  8  N(0,1), uniform routing
q2k        2048  4096   256  2048  8  N(0,1); down projection in Q2_K
q2k_dec..  1/64  4096   256  2048  8  the q2k layer with the decode1 / decode64 recipes
=========  ====  =====  ===  ====  =  ==========================================

The 4096-token prefill chunk is the distributed-prefill chunk of
"複数 Mac で 1 つのモデルを動かす: DwarfStar の TCP パイプライン分散推論を読む"
(§3, prefill as an assembly line); the few-token decode and the 64-token
micro-batch mirror the batched sessions of "DwarfStar実地分析" (§ローカルエージェント
と互換サーバーの使い分け).  The weights of decode1/decode64/prefill are one and
the same layer (weight seed 1).

Weight values ~ N(0, 0.02), encoded per 32-element block along the contraction
dimension: E8M0 scale s = largest integer with 6*2^s <= amax (amax = 0 -> 0),
codes = E2M1 round-to-nearest-even of v / 2^s saturating at +-6 (OCP
Microscaling Formats v1.0 value set; the nibble of element 2i is the low
nibble of byte i).

Randomness: ``torch.Generator`` on the target device, one generator per
(seed, tensor).  CPU and CUDA generators give different streams for the same
seed, so a run generates once and hands the same bytes to both sides.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = [
    "Workload", "WORKLOADS", "E2M1_GRID",
    "encode_mxfp4", "encode_q2k", "make_logits", "make_x",
    "make_layer_weights", "make_dense_weights", "make_inputs",
]

# E2M1 magnitudes for codes 0..7 (OCP MX v1.0, FP4 E2M1).
E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    f: int
    k: int
    seed: int          # seed for logits and x
    weight_seed: int   # seed for the expert weights
    routing: str       # "perm", "normal", "zipf"
    down: str = "mxfp4"  # or "q2k"

    @property
    def expert_bytes(self) -> int:
        """Bytes of one expert's stored weights (gate + up + down)."""
        gu = 2 * self.f * self.d * 17 // 32
        if self.down == "q2k":
            dn = self.d * (self.f // 256) * 84
        else:
            dn = self.d * self.f * 17 // 32
        return gu + dn


WORKLOADS = {
    "tiny": Workload("tiny", 4, 256, 8, 128, 2, 0, 0, "perm"),
    "decode1": Workload("decode1", 1, 4096, 256, 2048, 8, 1, 1, "normal"),
    "decode64": Workload("decode64", 64, 4096, 256, 2048, 8, 2, 1, "zipf"),
    "prefill": Workload("prefill", 4096, 4096, 256, 2048, 8, 3, 1, "normal"),
    "q2k": Workload("q2k", 2048, 4096, 256, 2048, 8, 4, 4, "normal", "q2k"),
    # profiling case: the prefill layer with 32 experts and 512 tokens, so each
    # expert still receives about 128 tokens (the per-expert GEMM shape of the
    # 4096-token chunk) while the device holds well under 1 GB
    "prefill_e32": Workload("prefill_e32", 512, 4096, 32, 2048, 8, 3, 1, "normal"),
    # the Q2_K layer (weight seed 4) at one token and at 64 tokens with a Zipf prior
    "q2k_decode1": Workload("q2k_decode1", 1, 4096, 256, 2048, 8, 1, 4, "normal", "q2k"),
    "q2k_decode64": Workload("q2k_decode64", 64, 4096, 256, 2048, 8, 2, 4, "zipf", "q2k"),
    # profiling cases of the few-token and Q2_K paths with fewer experts (the
    # per-expert shapes of the full workloads, a fraction of the device memory)
    "decode1_e32": Workload("decode1_e32", 1, 4096, 32, 2048, 8, 1, 1, "normal"),
    "decode64_e64": Workload("decode64_e64", 64, 4096, 64, 2048, 8, 2, 1, "zipf"),
    "q2k_e64": Workload("q2k_e64", 512, 4096, 64, 2048, 8, 4, 4, "normal", "q2k"),
}


def _gen(device, seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream * 7919 + 12345) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


# ---------------------------------------------------------------------------
# MXFP4 encoder (input preparation only)
# ---------------------------------------------------------------------------
def _mxfp4_block_exponent(amax: torch.Tensor) -> torch.Tensor:
    """Largest integer s with 6*2^s <= amax (0 where amax == 0), clamped to
    the E8M0 range [-127, 127].  Exact: amax = m*2^e with m in [0.5, 1);
    6*2^(e-3) = 0.75*2^e <= amax iff m >= 0.75."""
    m, e = torch.frexp(amax)
    s = torch.where(m >= 0.75, e - 3, e - 4)
    s = torch.where(amax > 0, s, torch.zeros_like(s))
    return s.clamp(-127, 127).to(torch.int32)


def _e2m1_rne_magnitude_code(a: torch.Tensor) -> torch.Tensor:
    """Round |v| (already divided by the block scale) to the nearest E2M1
    magnitude, ties to the code with an even mantissa bit, saturating at 6."""
    code = torch.zeros_like(a, dtype=torch.uint8)
    # (threshold, strict) pairs: value above threshold (or >= when the upper
    # neighbour is the even code) moves to the next code.
    steps = [
        (0.25, True),   # 0 | 0.5  : tie -> 0 (code 0 even)
        (0.75, False),  # 0.5 | 1  : tie -> 1 (code 2 even)
        (1.25, True),   # 1 | 1.5  : tie -> 1
        (1.75, False),  # 1.5 | 2  : tie -> 2
        (2.5, True),    # 2 | 3    : tie -> 2
        (3.5, False),   # 3 | 4    : tie -> 4
        (5.0, True),    # 4 | 6    : tie -> 4
    ]
    for thr, strict in steps:
        up = (a > thr) if strict else (a >= thr)
        code = code + up.to(torch.uint8)
    return code


def encode_mxfp4(w: torch.Tensor):
    """Encode fp32 ``w[..., K]`` (K % 32 == 0) blockwise along the last axis.

    Returns ``(codes uint8[..., K//2], scales uint8[..., K//32])``."""
    assert w.dtype == torch.float32 and w.shape[-1] % 32 == 0
    K = w.shape[-1]
    blocks = w.reshape(*w.shape[:-1], K // 32, 32)
    amax = blocks.abs().amax(dim=-1)
    s = _mxfp4_block_exponent(amax)
    v = torch.ldexp(blocks, (-s).unsqueeze(-1).to(torch.float32))
    mag = _e2m1_rne_magnitude_code(v.abs())
    neg = (v < 0) & (mag > 0)
    code = mag | (neg.to(torch.uint8) << 3)
    code = code.reshape(*w.shape[:-1], K // 2, 2)
    codes = code[..., 0] | (code[..., 1] << 4)
    scales = (s + 127).to(torch.uint8)
    return codes.contiguous(), scales.contiguous()


# ---------------------------------------------------------------------------
# Q2_K-style encoder (input preparation only)
# ---------------------------------------------------------------------------
def encode_q2k(w: torch.Tensor) -> torch.Tensor:
    """Encode fp32 ``w[..., K]`` (K % 256 == 0) into 84-byte super-blocks.

    Super-block layout (256 weights = 16 sub-blocks of 16):
      bytes  0..15  scales[j]: low nibble sc_j, high nibble m_j
      bytes 16..79  qs: weight i at byte 16 + i//4, bits 2*(i%4)
      bytes 80..81  fp16 d    (little endian)
      bytes 82..83  fp16 dmin (little endian)
    decoded weight = d*sc_j*q - dmin*m_j.

    Encoder (one plain choice; the layer only decodes): per sub-block
    lo = min(0, min w), hi = max(w), s_j = (hi - lo)/3, m_j = -lo;
    d = fp16(max_j s_j / 15), dmin = fp16(max_j m_j / 15);
    sc_j = clamp(rint(s_j/d), 0, 15), mq_j = clamp(rint(m_j/dmin), 0, 15);
    q = clamp(rint((w + dmin*mq_j) / (d*sc_j)), 0, 3) (0 where d*sc_j == 0).
    Returns uint8[..., K//256, 84]."""
    assert w.dtype == torch.float32 and w.shape[-1] % 256 == 0
    lead = w.shape[:-1]
    nsb = w.shape[-1] // 256
    sub = w.reshape(*lead, nsb, 16, 16).to(torch.float64)
    lo = torch.clamp(sub.amin(dim=-1), max=0.0)
    hi = sub.amax(dim=-1)
    s = (hi - lo) / 3.0
    m = -lo
    d16 = (s.amax(dim=-1) / 15.0).to(torch.float16)
    dm16 = (m.amax(dim=-1) / 15.0).to(torch.float16)
    d = d16.to(torch.float64).unsqueeze(-1)
    dm = dm16.to(torch.float64).unsqueeze(-1)
    sc = torch.where(d > 0, torch.round(s / torch.where(d > 0, d, torch.ones_like(d))),
                     torch.zeros_like(s)).clamp(0, 15)
    mq = torch.where(dm > 0, torch.round(m / torch.where(dm > 0, dm, torch.ones_like(dm))),
                     torch.zeros_like(m)).clamp(0, 15)
    step = (d * sc).unsqueeze(-1)
    off = (dm * mq).unsqueeze(-1)
    q = torch.where(step > 0, torch.round((sub + off) / torch.where(step > 0, step, torch.ones_like(step))),
                    torch.zeros_like(sub)).clamp(0, 3).to(torch.uint8)
    q = q.reshape(*lead, nsb, 64, 4)
    qs = q[..., 0] | (q[..., 1] << 2) | (q[..., 2] << 4) | (q[..., 3] << 6)
    scales = (sc.to(torch.uint8) | (mq.to(torch.uint8) << 4))
    dd = torch.stack([d16, dm16], dim=-1).contiguous().view(torch.uint8).reshape(*lead, nsb, 4)
    out = torch.cat([scales, qs, dd], dim=-1)
    assert out.shape[-1] == 84
    return out.contiguous()


# ---------------------------------------------------------------------------
# activations and router logits
# ---------------------------------------------------------------------------
def make_x(wl: Workload, device="cpu", T: Optional[int] = None) -> torch.Tensor:
    """x ~ N(0,1) rounded to bf16 (RNE), shape [T, d]."""
    T = wl.T if T is None else T
    g = _gen(device, wl.seed, 1)
    return torch.randn(T, wl.d, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def _break_ties(logits: torch.Tensor, g: torch.Generator) -> torch.Tensor:
    """Add pi(e)*2^-20 (pi a seeded permutation) to every row that holds an
    exact tie among its logits."""
    T, E = logits.shape
    srt, _ = logits.sort(dim=1)
    tied = (srt[:, 1:] == srt[:, :-1]).any(dim=1)
    if bool(tied.any()):
        pi = torch.randperm(E, generator=g, device=logits.device).to(torch.float32)
        logits = torch.where(tied.unsqueeze(1), logits + pi * 2.0 ** -20, logits)
    return logits


def make_logits(wl: Workload, device="cpu", T: Optional[int] = None) -> torch.Tensor:
    """Router logits fp32 [T, E] following the workload's recipe."""
    T = wl.T if T is None else T
    g = _gen(device, wl.seed, 2)
    E = wl.E
    if wl.routing == "perm":
        base = torch.stack([torch.randperm(E, generator=g, device=device) for _ in range(T)]).to(torch.float32)
        logits = base * 0.5 + 0.01 * torch.randn(T, E, generator=g, device=device)
    elif wl.routing == "normal":
        logits = torch.randn(T, E, generator=g, device=device)
    elif wl.routing == "zipf":
        pi = torch.randperm(E, generator=g, device=device)
        ranks = torch.arange(1, E + 1, device=device, dtype=torch.float64)
        p = ranks ** -1.1
        p = p / p.sum()
        prior = torch.log(p).to(torch.float32)[pi]  # expert e has rank pi[e]+1
        logits = torch.randn(T, E, generator=g, device=device) + prior.unsqueeze(0)
    else:
        raise ValueError(wl.routing)
    return _break_ties(logits.to(torch.float32).contiguous(), g)


# ---------------------------------------------------------------------------
# expert weights
# ---------------------------------------------------------------------------
def make_layer_weights(wl: Workload, device="cpu", experts: Optional[int] = None) -> dict:
    """Canonical stored weights of the layer.

    gate_codes/up_codes uint8[E, f, d/2], gate_scales/up_scales uint8[E, f, d/32];
    MXFP4 down: down_codes uint8[E, d, f/2], down_scales uint8[E, d, f/32];
    Q2_K down:  down_q2k uint8[E, d, f/256, 84].
    Generated expert by expert so peak memory stays at one fp32 matrix."""
    E = wl.E if experts is None else experts
    d, f = wl.d, wl.f
    out = {
        "gate_codes": torch.empty(E, f, d // 2, dtype=torch.uint8, device=device),
        "gate_scales": torch.empty(E, f, d // 32, dtype=torch.uint8, device=device),
        "up_codes": torch.empty(E, f, d // 2, dtype=torch.uint8, device=device),
        "up_scales": torch.empty(E, f, d // 32, dtype=torch.uint8, device=device),
    }
    if wl.down == "q2k":
        out["down_q2k"] = torch.empty(E, d, f // 256, 84, dtype=torch.uint8, device=device)
    else:
        out["down_codes"] = torch.empty(E, d, f // 2, dtype=torch.uint8, device=device)
        out["down_scales"] = torch.empty(E, d, f // 32, dtype=torch.uint8, device=device)
    gens = [_gen(device, wl.weight_seed, 100 + i) for i in range(3)]
    for e in range(E):
        wg = torch.randn(f, d, generator=gens[0], device=device) * 0.02
        out["gate_codes"][e], out["gate_scales"][e] = encode_mxfp4(wg)
        wu = torch.randn(f, d, generator=gens[1], device=device) * 0.02
        out["up_codes"][e], out["up_scales"][e] = encode_mxfp4(wu)
        wd = torch.randn(d, f, generator=gens[2], device=device) * 0.02
        if wl.down == "q2k":
            out["down_q2k"][e] = encode_q2k(wd)
        else:
            out["down_codes"][e], out["down_scales"][e] = encode_mxfp4(wd)
    return out


def make_dense_weights(wl: Workload, fs: int, device="cpu", router: bool = True) -> dict:
    """Original-precision (bf16) parts of the layer: router [E, d] with entries
    N(0, 1/d) (so that the logits of N(0,1) activations are about N(0, 1)) and
    a shared expert of intermediate size fs, gate/up [fs, d] and down [d, fs]
    with entries N(0, 0.02)."""
    out = {}
    g = _gen(device, wl.weight_seed, 200)
    if router:
        out["router"] = (torch.randn(wl.E, wl.d, generator=g, device=device) / math.sqrt(wl.d)).to(torch.bfloat16)
    if fs > 0:
        out["shared_gate"] = (torch.randn(fs, wl.d, generator=g, device=device) * 0.02).to(torch.bfloat16)
        out["shared_up"] = (torch.randn(fs, wl.d, generator=g, device=device) * 0.02).to(torch.bfloat16)
        out["shared_down"] = (torch.randn(wl.d, fs, generator=g, device=device) * 0.02).to(torch.bfloat16)
    return out


def make_inputs(wl: Workload, device="cpu", T: Optional[int] = None) -> dict:
    """Logits and x for one forward call."""
    return {"x": make_x(wl, device, T), "logits": make_logits(wl, device, T)}
