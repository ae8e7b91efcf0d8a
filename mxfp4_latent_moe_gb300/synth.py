"""Seeded synthetic inputs for the MXFP4 latent-MoE layer.

This module only draws random numbers in the shapes and distributions of the
layer's workloads; it holds none of the layer's arithmetic. Both the CUDA path
and the CPU oracle receive the same tensors from here.

Workloads (the layer of "Kimi K3.1 Pro on AMD Instinct GPUs", "Kimi K3.1 Pro at
a glance": 896 routed experts, top-16, intermediate 3,072 in a 3,584-wide
latent; MXFP4 weights with one E8M0 scale per 32 values):

  tiny                T=8,     d=256,  E=32,  k=4,  I=128
  decode_t64          T=64,    d=3584, E=896, k=16, I=3072
  decode_t512         T=512,   full dims
  prefill_skewed_t8192  T=8192, full dims, logits + 2*ln(1/rank_e) for a random
                      expert ranking (Zipf-like load)
  prefill_outlier_t32768 T=32768, full dims, 1% of x rows scaled by 64

Distributions: x ~ N(0,1) rounded to bf16; logits ~ N(0,1) fp32; weight codes
are uniform random bytes (two uniform E2M1 codes each, all 16 codes including
-0); weight scale codes uniform over the integers 118..122.

Draw order from one torch.Generator seeded with `seed` on `device`: x, logits,
expert ranking, outlier rows, w13 codes, w13 scales, w2 codes, w2 scales.
A given (seed, device type) always gives the same tensors; the CPU and CUDA
generators give different streams.
"""
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    E: int
    k: int
    I: int
    skew: bool = False          # add 2*ln(1/rank) per expert to the logits
    outlier_frac: float = 0.0   # fraction of x rows scaled by outlier_scale
    outlier_scale: float = 64.0


WORKLOADS = [
    Workload("tiny", T=8, d=256, E=32, k=4, I=128),
    Workload("decode_t64", T=64, d=3584, E=896, k=16, I=3072),
    Workload("decode_t512", T=512, d=3584, E=896, k=16, I=3072),
    Workload("prefill_skewed_t8192", T=8192, d=3584, E=896, k=16, I=3072, skew=True),
    Workload("prefill_outlier_t32768", T=32768, d=3584, E=896, k=16, I=3072,
             outlier_frac=0.01),
]
# Reduced cases of the same kernels for profiler captures (about 1 GB of
# weights, still far larger than the 129 MB L2): full d and I, 64 experts.
# At T = 1792 every expert holds 4 token tiles of 128 rows (448 routed rows
# on average, standard deviation 18), at T = 2304 five (576 on average, 21),
# as at T = 32,768 with 896 experts.
PROFILE_WORKLOADS = [
    Workload("ncu_decode_t64_e64", T=64, d=3584, E=64, k=16, I=3072),
    Workload("ncu_prefill_t2048_e64", T=2048, d=3584, E=64, k=16, I=3072),
    Workload("ncu_prefill_t1792_e64", T=1792, d=3584, E=64, k=16, I=3072),
    Workload("ncu_prefill_t2304_e64", T=2304, d=3584, E=64, k=16, I=3072),
]
BY_NAME = {w.name: w for w in WORKLOADS + PROFILE_WORKLOADS}


def workload(name_or_index):
    if isinstance(name_or_index, int):
        return WORKLOADS[name_or_index]
    return BY_NAME[name_or_index]


def full_dims(T):
    """T tokens at the full layer dims (d=3584, E=896, k=16, I=3072), N(0,1) logits."""
    return Workload("uniform_t%d" % T, T=T, d=3584, E=896, k=16, I=3072)


def shape(name, T=None, d=None, E=None, k=None, I=None, **kw):
    """A custom workload (test shapes)."""
    return Workload(name, T=T, d=d, E=E, k=k, I=I, **kw)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_activations(wl: Workload, seed=0, device="cpu", g=None):
    """x bf16 [T][d], logits fp32 [T][E] (draws 1-4 of the fixed order)."""
    g = g if g is not None else _gen(seed, device)
    T, d, E = wl.T, wl.d, wl.E
    x = torch.randn(T, d, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    logits = torch.randn(T, E, generator=g, device=device, dtype=torch.float32)
    if wl.skew:
        order = torch.randperm(E, generator=g, device=device)
        rank = torch.empty(E, dtype=torch.float32, device=device)
        rank[order] = torch.arange(1, E + 1, dtype=torch.float32, device=device)
        logits = logits + 2.0 * torch.log(1.0 / rank)[None, :]
    if wl.outlier_frac > 0 and T > 0:
        n_out = int(round(wl.outlier_frac * T))
        rows = torch.randperm(T, generator=g, device=device)[:n_out]
        x[rows] = (x[rows].float() * wl.outlier_scale).to(torch.bfloat16)
    return x, logits


def make_weights(wl: Workload, seed=0, device="cpu", g=None):
    """Canonical MXFP4 weights (draws 5-8 of the fixed order).

    w13 u8 [E][2I][d/2]: rows 0..I-1 gate (w1), rows I..2I-1 up (w3), two E2M1
    codes per byte, the even element in the low nibble.
    w13_s u8 [E][2I][d/32]: E8M0 scale codes, one per 32 consecutive inputs.
    w2 u8 [E][d][I/2], w2_s u8 [E][d][I/32]: the down projection, same packing.
    """
    g = g if g is not None else _gen(seed, device)
    E, d, I = wl.E, wl.d, wl.I
    u8 = torch.uint8
    w13 = torch.randint(0, 256, (E, 2 * I, d // 2), dtype=u8, generator=g, device=device)
    w13_s = torch.randint(118, 123, (E, 2 * I, d // 32), dtype=u8, generator=g, device=device)
    w2 = torch.randint(0, 256, (E, d, I // 2), dtype=u8, generator=g, device=device)
    w2_s = torch.randint(118, 123, (E, d, I // 32), dtype=u8, generator=g, device=device)
    return dict(w13=w13, w13_s=w13_s, w2=w2, w2_s=w2_s)


def make_layer(wl: Workload, seed=0, device="cpu"):
    """All inputs of one layer call in the fixed draw order."""
    g = _gen(seed, device)
    x, logits = make_activations(wl, g=g, device=device)
    weights = make_weights(wl, g=g, device=device)
    return dict(x=x, logits=logits, **weights)


@dataclass(frozen=True)
class BlockWorkload:
    """The composed block around the routed layer: hidden width, latent d,
    routed experts (E, k, I) and the shared experts' total intermediate width
    ("Kimi K3.1 Pro at a glance": hidden 7,168, latent 3,584, two shared
    experts; each shared expert 7,168 -> 3,072 -> 7,168)."""
    name: str
    T: int
    hidden: int
    d: int
    E: int
    k: int
    I: int
    shared_I: int

    @property
    def routed(self):
        return Workload(self.name + "_routed", T=self.T, d=self.d, E=self.E, k=self.k, I=self.I)


BLOCK_WORKLOADS = [
    BlockWorkload("block_decode_t64", T=64, hidden=7168, d=3584, E=896, k=16, I=3072,
                  shared_I=6144),
    BlockWorkload("block_prefill_t8192", T=8192, hidden=7168, d=3584, E=896, k=16, I=3072,
                  shared_I=6144),
]
BLOCK_BY_NAME = {w.name: w for w in BLOCK_WORKLOADS}


def block_workload(name):
    return BLOCK_BY_NAME[name]


def block_shape(name, T, hidden, d, E, k, I, shared_I):
    return BlockWorkload(name, T=T, hidden=hidden, d=d, E=E, k=k, I=I, shared_I=shared_I)


def _grid_bf16(shape_, scale, lo, hi, g, device):
    """Integers uniform in [lo, hi] times `scale` (a power of two), as bf16."""
    v = torch.randint(lo, hi + 1, shape_, generator=g, device=device, dtype=torch.int32)
    return (v.to(torch.float32) * scale).to(torch.bfloat16)


def make_block(bw: BlockWorkload, seed=0, device="cpu"):
    """All inputs of one block call. Draw order: h, w_down, w_router,
    w_shared13, w_out, then the routed experts' weights (as make_weights).

    Values sit on coarse power-of-two grids so that every product the block's
    BF16 GEMMs form before a rounding is exact in fp32: h = N(0,1) rounded to
    multiples of 1/8 and clamped to [-4, 4]; every BF16 weight an integer
    uniform in [-16, 16] times 2^-8. A dot product over 7,168 inputs is then a
    multiple of 2^-11 below 2^11 in magnitude (22 significant bits), so the
    router logits and the latent x are the same whatever the order of the
    fp32 additions: the routing decisions that depend on them cannot differ
    between two correct implementations."""
    g = _gen(seed, device)
    T, hd, d, E, Is = bw.T, bw.hidden, bw.d, bw.E, bw.shared_I
    h = (torch.randn(T, hd, generator=g, device=device) * 8).round().clamp(-32, 32) / 8
    out = dict(h=h.to(torch.bfloat16))
    out["w_down"] = _grid_bf16((d, hd), 2.0 ** -8, -16, 16, g, device)
    out["w_router"] = _grid_bf16((E, hd), 2.0 ** -8, -16, 16, g, device)
    out["w_shared13"] = _grid_bf16((2 * Is, hd), 2.0 ** -8, -16, 16, g, device)
    out["w_out"] = _grid_bf16((hd, d + Is), 2.0 ** -8, -16, 16, g, device)
    out.update(make_weights(bw.routed, g=g, device=device))
    return out


def random_e4m3_codes(shape_, seed=0, device="cpu", g=None):
    """Uniform finite E4M3 codes (magnitude codes 0x00..0x7E, either sign)."""
    g = g if g is not None else _gen(seed, device)
    mag = torch.randint(0, 0x7F, shape_, dtype=torch.uint8, generator=g, device=device)
    sign = torch.randint(0, 2, shape_, dtype=torch.uint8, generator=g, device=device) * 0x80
    return mag | sign


def random_scale_codes(shape_, lo=118, hi=122, seed=0, device="cpu", g=None):
    g = g if g is not None else _gen(seed, device)
    return torch.randint(lo, hi + 1, shape_, dtype=torch.uint8, generator=g, device=device)


def bf16_bits(t):
    """bf16 tensor -> its uint16 bit patterns as a numpy array (CPU)."""
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view("uint16")
