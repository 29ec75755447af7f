"""Seeded synthetic inputs for the block-scaled backward path.

This module builds the packed operands, scales, gradients and expert offsets that
both the CUDA library and the CPU oracle consume.  It does none of the backward
arithmetic (no decode, no scale application, no product): it only draws random
numbers and ENCODES them into the packed formats, the job the forward pass's
quantizer does before a backward ever runs.  Every tensor is drawn from its own
seeded ``torch.Generator`` on the requested device, so a given (config, seed,
device) always yields the same bytes.

Encoders (inputs only; the parity tests never compare them):
  * FP8 E4M3 with 128x128 blocks: scale_inv = amax / 448 per block (float32),
    codes = E4M3 nearest-even of w / scale_inv; an all-zero block gets
    scale_inv = 1.  (transformers PR #50031 stores E4M3 weights with float32
    ``weight_scale_inv`` blocks of 128x128; 448 is E4M3's max, AstrAI fp8.py.)
  * MXFP4: per 32 consecutive elements of a row, E8M0 exponent
    e = the least integer with 2^e >= amax / 6, byte = clamp(e + 127, 0, 254),
    codes = E2M1 nearest-even of x / 2^e; an all-zero block gets byte 0.
  * NVFP4: tensor scale t = amax_tensor / (6 * 448) (float32), per 16 elements an
    E4M3 block scale s = E4M3(amax_block / (6 t)), codes = E2M1 nearest-even of
    x / (s * t); a zero block scale gives zero codes.
  * E2M1 packing: element 2j in the low nibble of byte j, 2j+1 in the high one.
"""

from dataclasses import dataclass, field

import numpy as np
import torch

FMT_BF16 = 0
FMT_FP8 = 1
FMT_MXFP4 = 2
FMT_NVFP4 = 3
FMT_FP8_TENSOR = 4
FMT_E5M2_TENSOR = 5
FMT_NAMES = {FMT_BF16: "bf16", FMT_FP8: "fp8_e4m3_b128", FMT_MXFP4: "mxfp4", FMT_NVFP4: "nvfp4",
             FMT_FP8_TENSOR: "fp8_e4m3_tensor", FMT_E5M2_TENSOR: "fp8_e5m2_tensor"}


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn(shape, std, seed, device, dtype=torch.float32):
    g = _gen(device, seed)
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(dtype)


# ---------------------------------------------------------------- encoders
_E2M1_LOW_TIES = (0.25, 1.25, 2.5, 5.0)    # a tie here rounds down to the even code
_E2M1_HIGH_TIES = (0.75, 1.75, 3.5)        # a tie here rounds up to the even code


def e2m1_encode(a):
    """float tensor (already divided by its scale) -> E2M1 codes (uint8), nearest even, saturating."""
    mag = a.abs()
    code = torch.zeros(a.shape, dtype=torch.int32, device=a.device)
    for t in _E2M1_LOW_TIES:
        code += (mag > t).to(torch.int32)
    for t in _E2M1_HIGH_TIES:
        code += (mag >= t).to(torch.int32)
    code = code | ((a < 0).to(torch.int32) << 3)
    return code.to(torch.uint8)


def pack_fp4(codes):
    """uint8 codes [..., C] -> packed bytes [..., C/2] (even element in the low nibble)."""
    c = codes.to(torch.int32)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).to(torch.uint8)


def quantize_fp8_b128(w):
    """float32 [B,R,C] -> (E4M3 codes uint8 [B,R,C], scale_inv float32 [B,ceil(R/128),ceil(C/128)])."""
    B, R, C = w.shape
    Rb, Cb = -(-R // 128), -(-C // 128)
    pad = torch.zeros((B, Rb * 128, Cb * 128), dtype=torch.float32, device=w.device)
    pad[:, :R, :C] = w
    blocks = pad.view(B, Rb, 128, Cb, 128)
    amax = blocks.abs().amax(dim=(2, 4))
    scale_inv = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (blocks / scale_inv[:, :, None, :, None]).clamp(-448.0, 448.0)
    codes = q.to(torch.float8_e4m3fn).view(torch.uint8).reshape(B, Rb * 128, Cb * 128)[:, :R, :C]
    return codes.contiguous(), scale_inv.contiguous()


def quantize_fp8_tensor(w):
    """float32 [B,R,C] -> (E4M3 codes uint8 [B,R,C], scale_inv float32 [B]): one scale per
    batch entry (amax / 448; an all-zero entry gets 1)."""
    B = w.shape[0]
    amax = w.abs().reshape(B, -1).amax(dim=1)
    scale_inv = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (w / scale_inv[:, None, None]).clamp(-448.0, 448.0)
    return q.to(torch.float8_e4m3fn).view(torch.uint8).contiguous(), scale_inv.to(torch.float32).contiguous()


def quantize_mxfp4(x):
    """float32 [B,R,C] (C % 32 == 0) -> (packed uint8 [B,R,C/2], E8M0 uint8 [B,R,C/32])."""
    B, R, C = x.shape
    blocks = x.view(B, R, C // 32, 32)
    amax = blocks.abs().amax(dim=-1).to(torch.float64)
    m, k = torch.frexp(amax / 6.0)                  # amax/6 = m * 2^k, m in [0.5, 1)
    e = torch.where(m == 0.5, k - 1, k)
    b = torch.where(amax > 0, (e + 127).clamp(0, 254), torch.zeros_like(e))
    inv = torch.ldexp(torch.ones_like(amax), (127 - b).to(torch.float64))
    q = (blocks.to(torch.float64) * inv[..., None]).clamp(-6.0, 6.0).to(torch.float32)
    codes = e2m1_encode(q).view(B, R, C)
    return pack_fp4(codes).contiguous(), b.to(torch.uint8).contiguous()


def quantize_nvfp4(x):
    """float32 [B,R,C] (C % 16 == 0) -> (packed [B,R,C/2], E4M3 block scales [B,R,C/16], float32 [B])."""
    B, R, C = x.shape
    amax_t = x.abs().reshape(B, -1).amax(dim=1)
    t = torch.where(amax_t > 0, amax_t / (6.0 * 448.0), torch.ones_like(amax_t))
    blocks = x.view(B, R, C // 16, 16)
    amax_b = blocks.abs().amax(dim=-1)
    s = (amax_b / (6.0 * t[:, None, None])).clamp(max=448.0).to(torch.float8_e4m3fn)
    denom = s.to(torch.float32) * t[:, None, None]
    q = torch.where(denom[..., None] > 0, blocks / denom[..., None].clamp(min=1e-30),
                    torch.zeros_like(blocks)).clamp(-6.0, 6.0)
    codes = e2m1_encode(q).view(B, R, C)
    return pack_fp4(codes).contiguous(), s.view(torch.uint8).contiguous(), t.to(torch.float32).contiguous()


# ---------------------------------------------------------------- packed tensor bundle
@dataclass
class Packed:
    """A [batch, rows, cols] operand in one of the library's formats (cols contiguous)."""
    fmt: int
    data: torch.Tensor
    scale: torch.Tensor = None
    tensor_scale: torch.Tensor = None
    batch: int = 1
    rows: int = 0
    cols: int = 0
    meta: dict = field(default_factory=dict)

    def to(self, device):
        mv = lambda t: None if t is None else t.to(device)
        return Packed(self.fmt, mv(self.data), mv(self.scale), mv(self.tensor_scale),
                      self.batch, self.rows, self.cols, dict(self.meta))

    def numpy(self):
        """(data, scale, tensor_scale) as numpy arrays (BF16 data as uint16 bits)."""
        d = self.data.detach().cpu()
        d = d.view(torch.int16).numpy().view(np.uint16) if d.dtype == torch.bfloat16 else d.numpy()
        s = None if self.scale is None else self.scale.detach().cpu().numpy()
        ts = None if self.tensor_scale is None else self.tensor_scale.detach().cpu().numpy()
        return d, s, ts


def quantize(fmt, x):
    """float32 [B,R,C] -> Packed in format ``fmt``."""
    B, R, C = x.shape
    if fmt == FMT_BF16:
        return Packed(fmt, x.to(torch.bfloat16).contiguous(), None, None, B, R, C)
    if fmt == FMT_FP8:
        d, s = quantize_fp8_b128(x)
        return Packed(fmt, d, s, None, B, R, C)
    if fmt == FMT_FP8_TENSOR:
        d, s = quantize_fp8_tensor(x)
        return Packed(fmt, d, s, None, B, R, C)
    if fmt == FMT_MXFP4:
        d, s = quantize_mxfp4(x)
        return Packed(fmt, d, s, None, B, R, C)
    if fmt == FMT_NVFP4:
        d, s, t = quantize_nvfp4(x)
        return Packed(fmt, d, s, t, B, R, C)
    raise ValueError(fmt)


def make_packed(fmt, batch, rows, cols, std, seed, device, chunk_rows=None):
    """Draw N(0, std) values [batch, rows, cols] and encode them, one batch entry at a time."""
    if fmt == FMT_BF16:
        return quantize(fmt, randn((batch, rows, cols), std, seed, device))
    parts = []
    for b in range(batch):
        x = randn((1, rows, cols), std, seed * 1000003 + b, device)
        parts.append(quantize(fmt, x))
        del x
    cat = lambda ts: None if ts[0] is None else torch.cat(ts, dim=0).contiguous()
    return Packed(fmt, cat([p.data for p in parts]), cat([p.scale for p in parts]),
                  cat([p.tensor_scale for p in parts]), batch, rows, cols)


def random_codes(fmt, batch, rows, cols, seed, device="cpu", scale_kind="random"):
    """Packed operand whose data bytes are uniform over all 256 values (code coverage).

    scale_kind: "random" (moderate positive scales), "edge" (extreme scales:
    E8M0 bytes 0/1/126/127/128/254, tiny and huge float32 scale_inv, E4M3
    subnormal block scales), "nan" (a few NaN scales) or "finite" (scales whose
    products with every code stay finite but are often not BF16 numbers or are
    subnormal: E8M0 bytes up to 200, float32 scale_inv with full mantissas over a
    wide exponent range, NVFP4 tensor scales from 1e-30 to 1e30; FP8 NaN codes are
    replaced by 448 so that every decoded value is finite).
    """
    g = _gen(device, seed)
    fp8 = fmt in (FMT_FP8, FMT_FP8_TENSOR, FMT_E5M2_TENSOR)
    nbytes = cols if fp8 else cols // 2
    data = torch.randint(0, 256, (batch, rows, nbytes), generator=g, device=device, dtype=torch.int32).to(torch.uint8)
    if fmt == FMT_E5M2_TENSOR and scale_kind == "finite":
        data = torch.where((data & 0x7C) == 0x7C, data - 4, data)   # S.11111.mm (inf, NaN) -> S.11110.mm
    elif fp8 and scale_kind == "finite":
        data = torch.where((data & 0x7F) == 0x7F, data - 1, data)   # S.1111.111 (NaN) -> S.1111.110 (448)
    ts = None
    if fp8:
        shape = (batch, -(-rows // 128), -(-cols // 128)) if fmt == FMT_FP8 else (batch,)
        s = torch.rand(shape, generator=g, device=device) + 0.5
        if scale_kind == "finite":
            # |code| <= 448 and scale < 2^117 keep every product below the BF16 maximum
            mant = torch.rand(shape, generator=g, device=device) + 1.0
            exps = torch.tensor([-137, -134, -131, -128, -125, -121, -60, -7, -3, 0, 5, 40, 100,
                                 100 if fmt == FMT_E5M2_TENSOR else 116],   # E5M2 codes reach 2^15.8
                                dtype=torch.float32, device=device)
            ex = exps[torch.randint(0, exps.numel(), shape, generator=g, device=device)]
            s = mant * torch.pow(2.0, ex)
        elif scale_kind == "edge":
            pool = torch.tensor([2.0 ** -130, 1e-40, 3.0e-39, 1.0, 0.1, 2.0 ** 7, 2.0 ** 8, 300.0,
                                 3.0e38, 1.17e-38, 2.0 ** -126, 7.0e-3], device=device)
            s = pool[torch.randint(0, pool.numel(), shape, generator=g, device=device)]
        elif scale_kind == "nan":
            s = s.masked_fill(torch.rand(shape, generator=g, device=device) < 0.2, float("nan"))
        scale = s.to(torch.float32)
    elif fmt == FMT_MXFP4:
        shape = (batch, rows, cols // 32)
        if scale_kind == "finite":
            pool = torch.tensor([0, 1, 2, 100, 127, 128, 129, 130, 150, 180, 200], device=device)
            scale = pool[torch.randint(0, pool.numel(), shape, generator=g, device=device)].to(torch.uint8)
        elif scale_kind == "edge":
            pool = torch.tensor([0, 1, 126, 127, 128, 129, 142, 143, 200, 254], device=device)
            scale = pool[torch.randint(0, pool.numel(), shape, generator=g, device=device)].to(torch.uint8)
        elif scale_kind == "nan":
            scale = torch.randint(100, 150, shape, generator=g, device=device).to(torch.uint8)
            scale = scale.masked_fill(torch.rand(shape, generator=g, device=device) < 0.2, 255)
        else:
            scale = torch.randint(110, 140, shape, generator=g, device=device).to(torch.uint8)
    elif fmt == FMT_NVFP4:
        shape = (batch, rows, cols // 16)
        if scale_kind == "finite":
            scale = torch.randint(0, 0x7F, shape, generator=g, device=device).to(torch.uint8)   # finite E4M3
            scale = scale | (torch.randint(0, 2, shape, generator=g, device=device).to(torch.uint8) << 7)
            tsv = torch.tensor([1e-30, 2.0 ** -120, 0.3712, 1e30, 7.3e-5, 3.1], device=device)
            ts = tsv[torch.arange(batch, device=device) % tsv.numel()].to(torch.float32)
        elif scale_kind == "edge":
            scale = torch.randint(0, 256, shape, generator=g, device=device).to(torch.uint8)
            tsv = torch.tensor([1e-30, 2.0 ** -120, 1.0, 3.0e35][:batch] + [0.5] * max(0, batch - 4), device=device)
            ts = tsv[:batch].to(torch.float32)
        elif scale_kind == "nan":
            scale = torch.randint(0, 256, shape, generator=g, device=device).to(torch.uint8)  # includes 0x7F/0xFF NaNs
        else:
            scale = torch.randint(0x20, 0x60, shape, generator=g, device=device).to(torch.uint8)
        if ts is None:
            ts = (torch.rand((batch,), generator=g, device=device) * 0.01 + 1e-3).to(torch.float32)
    else:
        raise ValueError(fmt)
    return Packed(fmt, data.contiguous(), scale.contiguous(), None if ts is None else ts.contiguous(),
                  batch, rows, cols)


# ---------------------------------------------------------------- expert routing
def offsets_from_counts(counts):
    """Cumulative END offsets (int32, no leading zero), as the grouped matmul takes them."""
    return np.cumsum(np.asarray(counts, dtype=np.int64)).astype(np.int32)


def zipf_counts(S, E, s, seed, force_empty=(0, 31, 63)):
    """Token counts per expert: Multinomial(S, p_r ~ r^-s), ranks permuted, given experts emptied.

    The emptied experts' tokens move to the largest expert, so the total stays S.
    """
    rng = np.random.default_rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    by_rank = rng.multinomial(S, p)
    counts = np.empty(E, dtype=np.int64)
    counts[rng.permutation(E)] = by_rank
    moved = 0
    for e in force_empty:
        if e < E:
            moved += counts[e]
            counts[e] = 0
    counts[int(np.argmax(counts))] += moved
    return counts


def dirichlet_counts(S, E, alpha, seed):
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.full(E, alpha, dtype=np.float64))
    return rng.multinomial(S, p).astype(np.int64)


# ---------------------------------------------------------------- the five workloads
CONFIG_NAMES = {
    1: "fp8_linear_tiny_M64_N128_K256",
    2: "mxfp4_linear_4096x4096x4096",
    3: "nvfp4_ffn_M8192_N14336_K5120",
    4: "fp8_grouped_dgrad_E64_S16384_N2816_K2048",
    5: "mxfp4_grouped_E128_S32768_N2048_K7168",
}


def make_config(n, device="cpu", seed=0, small_m=16, experts=None, rows=None):
    """Inputs of workload ``n`` (1..5) on ``device``; returns a dict of tensors and sizes.

    Keys: ``G`` (bf16 grad_out), ``W`` (Packed, [E or 1, N, K]), ``X`` (Packed or None,
    [1, M, K]), ``offsets`` (int32 numpy, grouped only), sizes M/S, N, K, E, and for
    workload 2 ``G_small`` (bf16 [small_m, N]).  ``experts`` (grouped workloads only)
    scales the workload down to that many experts with the same tokens per expert and
    the same routing law (a smaller case of the same kernels, e.g. for profiling).
    ``rows`` (workload 4 only) keeps the 64 expert weights and routes that many grad_out
    rows instead of 16384 under the same law: a decode-sized batch.
    """
    base = seed * 100
    if n == 1:
        M, N, K = 64, 128, 256
        X = make_packed(FMT_BF16, 1, M, K, 1.0, base + 1, device)
        W = make_packed(FMT_FP8, 1, N, K, 0.02, base + 2, device)
        G = randn((M, N), 1.0, base + 3, device, torch.bfloat16)
        return dict(name=CONFIG_NAMES[n], M=M, N=N, K=K, E=1, G=G, W=W, X=X, grouped=False)
    if n == 2:
        M = N = K = 4096
        X = make_packed(FMT_MXFP4, 1, M, K, 1.0, base + 1, device)
        W = make_packed(FMT_MXFP4, 1, N, K, 1.0, base + 2, device)
        G = randn((M, N), 1.0, base + 3, device, torch.bfloat16)
        Gs = randn((small_m, N), 1.0, base + 4, device, torch.bfloat16)
        return dict(name=CONFIG_NAMES[n], M=M, N=N, K=K, E=1, G=G, W=W, X=X, G_small=Gs, grouped=False)
    if n == 3:
        M, N, K = 8192, 14336, 5120
        X = make_packed(FMT_NVFP4, 1, M, K, 0.02, base + 1, device)
        W = make_packed(FMT_NVFP4, 1, N, K, 0.02, base + 2, device)
        G = randn((M, N), 1e-2, base + 3, device, torch.bfloat16)
        return dict(name=CONFIG_NAMES[n], M=M, N=N, K=K, E=1, G=G, W=W, X=X, grouped=False)
    if n == 4:
        E, S, N, K = 64, 16384, 2816, 2048
        if experts:
            E, S = experts, S * experts // E
        if rows:
            S = rows
        counts = zipf_counts(S, E, 1.1, base + 5, force_empty=[e for e in (0, 31, 63) if e < E])
        W = make_packed(FMT_FP8, E, N, K, 0.02, base + 2, device)
        G = randn((S, N), 1.0, base + 3, device, torch.bfloat16)
        name = (f"fp8_grouped_dgrad_decode_E{E}_S{S}_N{N}_K{K}" if rows
                else CONFIG_NAMES[n] if E == 64 else f"fp8_grouped_dgrad_E{E}_S{S}_N{N}_K{K}")
        return dict(name=name, M=S, N=N, K=K, E=E, G=G, W=W, X=None,
                    offsets=offsets_from_counts(counts), grouped=True)
    if n == 5:
        E, S, N, K = 128, 32768, 2048, 7168
        if experts:
            E, S = experts, S * experts // E
        counts = dirichlet_counts(S, E, 0.3, base + 5)
        X = make_packed(FMT_MXFP4, 1, S, K, 1.0, base + 1, device)
        W = make_packed(FMT_MXFP4, E, N, K, 1.0, base + 2, device)
        G = randn((S, N), 1.0, base + 3, device, torch.bfloat16)
        name = CONFIG_NAMES[n] if E == 128 else f"mxfp4_grouped_E{E}_S{S}_N{N}_K{K}"
        return dict(name=name, M=S, N=N, K=K, E=E, G=G, W=W, X=X,
                    offsets=offsets_from_counts(counts), grouped=True)
    raise ValueError(n)


def bf16_numpy(t):
    """BF16 torch tensor -> numpy uint16 bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
