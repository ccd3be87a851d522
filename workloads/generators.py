"""Counter-based random numbers that agree between CPU and CUDA.

Every value is a pure function of (seed, stream, element index).  The hash is
the 32-bit MurmurHash3 finaliser (fmix32), applied to the low and high halves
of the 64-bit element counter under two stream keys.  Integer products are
split into 16-bit halves so no intermediate ever leaves the int64 range, which
keeps the integer part bit-identical on every torch backend.  Uniforms are
(h + 0.5) / 2^32; normals use the Box-Muller transform in float64.  The float64
transcendental functions may differ by an ulp between CPU libm and CUDA, which
changes a value rounded to bf16/fp32 with probability ~2^-40 per element; for
exact agreement the harness generates on one device and copies.
"""
import torch

M32 = 0xFFFFFFFF
_C1 = 0x85EBCA6B
_C2 = 0xC2B2AE35


def _mul32(h, c):
    """(h * c) mod 2^32 for int64 tensors with 0 <= h < 2^32 and a 32-bit constant c."""
    lo = c & 0xFFFF
    hi = c >> 16
    return (h * lo + (((h * hi) & 0xFFFF) << 16)) & M32


def _fmix32(h):
    h = h ^ (h >> 16)
    h = _mul32(h, _C1)
    h = h ^ (h >> 13)
    h = _mul32(h, _C2)
    h = h ^ (h >> 16)
    return h


def _fmix32_int(h):
    h &= M32
    h ^= h >> 16
    h = (h * _C1) & M32
    h ^= h >> 13
    h = (h * _C2) & M32
    h ^= h >> 16
    return h


def _keys(seed, stream):
    k0 = _fmix32_int((seed * 0x9E3779B1 + 0x7F4A7C15) & M32)
    k1 = _fmix32_int((stream * 0x85EBCA77 + k0 + 0x165667B1) & M32)
    k2 = _fmix32_int(k1 ^ 0x27D4EB2F)
    return k1, k2


def _hash_bits(seed, stream, offset, n, device, salt=0):
    idx = torch.arange(n, dtype=torch.int64, device=device) + int(offset)
    lo = idx & M32
    hi = idx >> 32
    k1, k2 = _keys(seed, stream * 2 + salt)
    h = _fmix32(lo ^ k1)
    h = _fmix32(h ^ ((hi + k2) & M32))
    return h


def counter_uniform(seed, stream, n, offset=0, device="cpu"):
    """n uniforms in (0, 1) as float64, element i keyed by (seed, stream, offset + i)."""
    h = _hash_bits(seed, stream, offset, n, device, salt=0)
    return (h.to(torch.float64) + 0.5) * (1.0 / 4294967296.0)


def counter_normal(seed, stream, n, offset=0, device="cpu"):
    """n standard normals as float64 (Box-Muller on two independent hash streams)."""
    u1 = counter_uniform(seed, stream, n, offset, device)
    h2 = _hash_bits(seed, stream, offset, n, device, salt=1)
    u2 = (h2.to(torch.float64) + 0.5) * (1.0 / 4294967296.0)
    return torch.sqrt(-2.0 * torch.log(u1)) * torch.cos(6.283185307179586 * u2)


def to_dtype_exact(t64, dtype):
    """Round a float64 tensor to the workload dtype ("f32" or "bf16").

    Returns a tensor of that torch dtype; widening it back to float64 is exact, so
    the oracle and the GPU path see the same input values."""
    if dtype == "f32":
        return t64.to(torch.float32)
    if dtype == "bf16":
        return t64.to(torch.float32).to(torch.bfloat16)
    raise ValueError(f"unknown dtype {dtype!r}")
