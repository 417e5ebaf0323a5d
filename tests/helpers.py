"""Shared test helpers: tolerance check for the GEMM, exhaustive bf16
plantings for the quantisers, and the library build fixture."""
from __future__ import annotations

import numpy as np
import torch

import oracle.fp8_oracle as O

# GEMM tolerance (reading of the stated bound for a bf16 output): relative
# Frobenius error <= 4e-3, and per element
#     |err| <= 1e-2 * rms(C_ref) + 2^-8 * |C_ref|
# where the second term is the half-ulp of bf16 at |C_ref| (the output is
# rounded to bf16, which alone exceeds 1e-2*rms for |C| above ~4 rms).
REL_FROB = 4e-3
ABS_RMS = 1e-2
BF16_HALF_ULP_REL = 2.0 ** -8


def gemm_errors(c_gpu: np.ndarray, c_ref: np.ndarray) -> dict:
    c_gpu = np.asarray(c_gpu, np.float64)
    c_ref = np.asarray(c_ref, np.float64)
    err = np.abs(c_gpu - c_ref)
    rms = float(np.sqrt(np.mean(c_ref ** 2))) if c_ref.size else 0.0
    fro = float(np.linalg.norm(c_ref))
    bound = ABS_RMS * rms + BF16_HALF_ULP_REL * np.abs(c_ref)
    return {
        "rel_frob": float(np.linalg.norm(c_gpu - c_ref) / fro) if fro > 0 else float(np.linalg.norm(c_gpu)),
        "max_err_over_rms": float(err.max() / rms) if rms > 0 and err.size else 0.0,
        "violations": int(np.sum(err > bound)),
        "literal_violations": int(np.sum(err > ABS_RMS * rms)),
        "nonfinite": int(np.sum(~np.isfinite(c_gpu))),
        "n": int(err.size),
    }


def assert_gemm_close(c_gpu, c_ref, what=""):
    e = gemm_errors(c_gpu, c_ref)
    assert e["nonfinite"] == 0, (what, e)
    assert e["rel_frob"] <= REL_FROB, (what, e)
    assert e["violations"] == 0, (what, e)
    return e


def bf16_to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def finite_bf16_values() -> np.ndarray:
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = O.bf16_bits_to_f32(bits)
    return f[np.isfinite(f)]


def amax_sweep(step: int = 7) -> np.ndarray:
    """Planted amax values: bf16 binades from the smallest subnormal upward
    (every `step`-th), each with mantissas 1.0, 1.75, just above 1.75 and a
    pseudo-random one (the pow2 rule switches at 1.75)."""
    out = []
    rng = np.random.Generator(np.random.PCG64(77))
    for e in range(-133, 128, step):
        for frac in (0x00, 0x60, 0x61, int(rng.integers(0, 128))):
            if e < -126:          # bf16 subnormal: value = m * 2^-133
                v = np.float32(2.0 ** e)
            else:
                v = np.float32((1 + frac / 128) * 2.0 ** e)
            out.append(v)
    a = torch.from_numpy(np.array(out, np.float32)).to(torch.bfloat16).float().numpy()
    return np.unique(a[np.isfinite(a) & (a > 0)])


def planted_rows(amaxes: np.ndarray, block: int, per_row_blocks: int, seed: int = 5) -> np.ndarray:
    """Rows of blocks of `block` values.  For each planted amax, every finite
    bf16 x with |x| <= amax appears in some block whose largest magnitude is
    exactly amax (the amax itself sits at a random position, random sign)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    f = finite_bf16_values()
    blocks = []
    for a in amaxes:
        vals = f[np.abs(f) <= a]
        vals = vals[rng.permutation(vals.size)]
        n = block - 1
        # repeat cyclically up to a whole number of blocks (small amax values
        # have fewer candidates than one block holds)
        vals = np.resize(vals, ((vals.size + n - 1) // n) * n)
        chunks = vals.reshape(-1, n)
        amax_col = np.where(rng.integers(0, 2, (chunks.shape[0], 1)) == 1, a, -a).astype(np.float32)
        blk = np.concatenate([amax_col, chunks], axis=1)
        idx = np.argsort(rng.random(blk.shape), axis=1)
        blocks.append(np.take_along_axis(blk, idx, axis=1))
    allb = np.concatenate(blocks, axis=0)
    allb = np.resize(allb, (((allb.shape[0] + per_row_blocks - 1) // per_row_blocks) * per_row_blocks,
                            allb.shape[1]))
    return allb.reshape(-1, per_row_blocks * block).astype(np.float32)
