"""Seeded synthetic inputs for the packed Q4_K matmul: weights, activations, shapes.

This module is shared by the tests, the benchmark and the smoke check, on both
sides of the parity check (the CPU oracle and the GPU library). It holds none of
the method's arithmetic: it only draws bytes and normal deviates.

Generator: SplitMix64 (S. Vigna's published 64-bit mixer) used counter-style,
``value(seed, i) = mix(seed + (i + 1) * 0x9E3779B97F4A7C15 mod 2**64)``. Being a
pure function of (seed, i) it is evaluated identically, and independently, on
the host and on the GPU with plain torch int64 tensor ops, so a test can rebuild
any sampled row of a multi-GB weight set on the host without copying it back.

Super-block g of a matrix (g = n * K/256 + b) takes stream values 19g .. 19g+18:
  value 0  bits 40..63 -> u_d, bits 16..39 -> u_dmin   (24-bit uniforms in [0,1))
           d = fp16(fp32(0.001) + fp32(0.019) * u)     (fp32 ops, then fp16 RNE),
           so d, dmin are uniform in [1e-3, 2e-2]
  value 1  bytes 0..7 -> scale bytes s[0..7]           (uniform 0..255)
  value 2  bytes 0..3 -> scale bytes s[8..11]
  values 3..18 -> the 128 qs bytes (two uniform 0..15 nibbles per byte)
Bytes of a 64-bit value are taken little-endian.

Activations: X[m, k] uses values 2e and 2e+1 (e = m*K + k) of the X stream:
Box-Muller in float64, z = sqrt(-2 ln u1) * cos(2 pi u2) with
u1 = (v >> 11 + 1) * 2**-53, u2 = (v' >> 11) * 2**-53, then rounded to fp32
(and from fp32 to bf16 with RNE for bf16 activations). X is always drawn on the
host and copied to the device, so both sides see the same bits.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
C1 = 0xBF58476D1CE4E5B9
C2 = 0x94D049BB133111EB
VALUES_PER_BLOCK = 19
BLOCK_BYTES = 144
BLOCK_WEIGHTS = 256
SEED_BASE = 0x51344B00


def _s64(v: int) -> int:
    v &= MASK64
    return v - (1 << 64) if v >= (1 << 63) else v


def splitmix64_py(seed: int, i: int) -> int:
    """Reference scalar evaluation (Python big ints): value i of stream ``seed``."""
    z = (seed + (i + 1) * GAMMA) & MASK64
    z = ((z ^ (z >> 30)) * C1) & MASK64
    z = ((z ^ (z >> 27)) * C2) & MASK64
    return z ^ (z >> 31)


def _srl(z: torch.Tensor, s: int) -> torch.Tensor:
    # logical right shift on int64 (torch's >> is arithmetic)
    return (z >> s) & ((1 << (64 - s)) - 1)


def _mix(z: torch.Tensor) -> torch.Tensor:
    z = (z ^ _srl(z, 30)) * _s64(C1)
    z = (z ^ _srl(z, 27)) * _s64(C2)
    return z ^ _srl(z, 31)


def stream(seed: int, start: int, count: int, device="cpu") -> torch.Tensor:
    """Values start .. start+count-1 of stream ``seed`` as int64 (two's complement)."""
    i = torch.arange(start + 1, start + count + 1, dtype=torch.int64, device=device)
    z = i * _s64(GAMMA) + _s64(seed)
    return _mix(z)


def _fp16_uniform(bits24: torch.Tensor) -> torch.Tensor:
    u = bits24.to(torch.float32) * (2.0 ** -24)          # exact
    span = torch.tensor(0.019, dtype=torch.float32, device=u.device)
    lo = torch.tensor(0.001, dtype=torch.float32, device=u.device)
    return torch.add(torch.mul(u, span), lo).to(torch.float16)


def blocks(seed: int, g0: int, nblk: int, device="cpu") -> torch.Tensor:
    """Super-blocks g0 .. g0+nblk-1 of stream ``seed`` as uint8 [nblk, 144]."""
    r = stream(seed, VALUES_PER_BLOCK * g0, VALUES_PER_BLOCK * nblk, device)
    r = r.view(nblk, VALUES_PER_BLOCK)
    r0 = r[:, 0]
    d = _fp16_uniform(_srl(r0, 40))
    dmin = _fp16_uniform((r0 >> 16) & 0xFFFFFF)
    d_b = d.view(torch.int16).view(torch.uint8).view(nblk, 2)
    dm_b = dmin.view(torch.int16).view(torch.uint8).view(nblk, 2)
    rest = r[:, 1:].contiguous().view(torch.uint8).view(nblk, 8 * (VALUES_PER_BLOCK - 1))
    s_lo = rest[:, 0:8]
    s_hi = rest[:, 8:12]
    qs = rest[:, 16:144]
    return torch.cat([d_b, dm_b, s_lo, s_hi, qs], dim=1)


def weight_rows(seed: int, N: int, K: int, row0: int = 0, nrows: int | None = None,
                device="cpu", chunk_blocks: int = 1 << 21,
                out: torch.Tensor | None = None) -> torch.Tensor:
    """Packed Q4_K rows row0 .. row0+nrows-1 of an N x K matrix: uint8 [nrows, K/256*144]."""
    if K % BLOCK_WEIGHTS:
        raise ValueError("K must be a multiple of 256")
    KB = K // BLOCK_WEIGHTS
    nrows = N - row0 if nrows is None else nrows
    if out is None:
        out = torch.empty((nrows, KB * BLOCK_BYTES), dtype=torch.uint8, device=device)
    rows_per = max(1, chunk_blocks // KB)
    for r in range(0, nrows, rows_per):
        nr = min(rows_per, nrows - r)
        b = blocks(seed, (row0 + r) * KB, nr * KB, device)
        out[r:r + nr].copy_(b.view(nr, KB * BLOCK_BYTES))
    return out


def weight_sample_rows(seed: int, N: int, K: int, rows) -> torch.Tensor:
    """Host bytes of an arbitrary set of rows (uint8 [len(rows), K/256*144])."""
    return torch.stack([weight_rows(seed, N, K, int(n), 1)[0] for n in rows])


def activations(seed: int, M: int, K: int, dtype=torch.float32) -> torch.Tensor:
    """Host activations X [M, K], N(0,1), fp32 or bf16 (see module docstring)."""
    n = M * K
    v = stream(seed, 0, 2 * n, "cpu").view(n, 2)
    u1 = (_srl(v[:, 0], 11) + 1).to(torch.float64) * (2.0 ** -53)
    u2 = _srl(v[:, 1], 11).to(torch.float64) * (2.0 ** -53)
    z = torch.sqrt(-2.0 * torch.log(u1)) * torch.cos((2.0 * math.pi) * u2)
    x = z.to(torch.float32).view(M, K)
    if dtype == torch.bfloat16:
        return x.to(torch.bfloat16)
    if dtype != torch.float32:
        raise ValueError("activations are fp32 or bf16")
    return x


# --------------------------------------------------------------------------
# Workload shapes: synthetic weight sets shaped like the models the pages run
# packed (Llama-3.2 / Orpheus on the rlx-llama32 page, the Qwen3 family on the
# rlx-qwen3 page). Random weights; no checkpoint is read.
# --------------------------------------------------------------------------

MATRIX_INDEX = {"q_proj": 0, "k_proj": 1, "v_proj": 2, "o_proj": 3,
                "gate_proj": 4, "up_proj": 5, "down_proj": 6, "lm_head": 7}


def weight_seed(workload: int, layer: int, matrix: str) -> int:
    return SEED_BASE + 1000 * workload + 16 * layer + MATRIX_INDEX[matrix]


def x_seed(workload: int, K: int, M: int) -> int:
    return SEED_BASE + 1000 * workload + 15 + (K << 20) + (M << 40)


@dataclass
class Workload:
    index: int
    name: str
    layer_shapes: list            # [(matrix, N, K)] per layer
    layers: int
    extra: list = field(default_factory=list)   # [(matrix, N, K)] once (lm_head)
    decode_m: tuple = ()
    prefill_m: tuple = ()
    x_dtypes: tuple = ("f32",)

    def matrices(self):
        """[(layer, matrix, N, K)] in sweep order."""
        out = [(layer, m, n, k) for layer in range(self.layers)
               for (m, n, k) in self.layer_shapes]
        out += [(self.layers, m, n, k) for (m, n, k) in self.extra]
        return out

    def packed_bytes(self) -> int:
        return sum(n * k // BLOCK_WEIGHTS * BLOCK_BYTES for (_, _, n, k) in self.matrices())


def _llama_like(q, kv, inter):
    return [("q_proj", q, q), ("k_proj", kv, q), ("v_proj", kv, q), ("o_proj", q, q),
            ("gate_proj", inter, q), ("up_proj", inter, q), ("down_proj", q, inter)]


WORKLOADS = {
    0: Workload(0, "tiny-256x512", [("q_proj", 256, 512)], 1, decode_m=(1, 4)),
    1: Workload(1, "llama-3.2-1b-shaped decode, 16 layers", _llama_like(2048, 512, 8192), 16,
                decode_m=(1,)),
    2: Workload(2, "llama-3.2-3b-shaped decode, 28 layers + lm_head",
                _llama_like(3072, 1024, 8192), 28, extra=[("lm_head", 128256, 3072)],
                decode_m=(1, 4, 16), x_dtypes=("f32", "bf16")),
    3: Workload(3, "qwen3-8b-shaped chunked prefill, 36 layers",
                _llama_like(4096, 1024, 12288), 36, prefill_m=(32, 512, 1024),
                x_dtypes=("bf16",)),
    4: Workload(4, "qwen3-14b-shaped sweep, 40 layers", _llama_like(5120, 1024, 17408), 40,
                decode_m=(1, 2, 4, 8, 16), prefill_m=(2048,), x_dtypes=("f32", "bf16")),
}
