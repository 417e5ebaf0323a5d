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


def weight_block_rows(w: torch.Tensor, nbs, pow2: bool = False):
    """Oracle 128x128 quantisation of the 128-row blocks `nbs` of a bf16
    weight [N, K] (a block row's tiles depend on nothing outside it).
    Returns (rows, q, s): the weight rows covered, their codes [len(rows), K]
    and scales [len(nbs), K/128]."""
    nbs = np.asarray(sorted(set(int(n) for n in nbs)))
    rows = np.concatenate([np.arange(nb * 128, (nb + 1) * 128) for nb in nbs])
    q, s = O.quant_weight_128x128(bf16_to_np(w[torch.from_numpy(rows)]), pow2)
    return rows, q, s


def sample_block_rows(N: int, count: int, seed: int):
    """`count` distinct 128-row blocks of an N-row weight, always including
    the first and the last."""
    nb = N // 128
    rng = np.random.Generator(np.random.PCG64(seed))
    pick = rng.choice(nb, min(count, nb), replace=False)
    return np.unique(np.concatenate([pick, [0, nb - 1]]))


def weight_block_cols(w: torch.Tensor, kbs, pow2: bool = False):
    """Oracle 128x128 quantisation of the 128-column blocks `kbs` of a bf16
    weight [N, K] (a block column's tiles depend on nothing outside it).
    Returns (cols, q [N, len(cols)], s [N/128, len(kbs)])."""
    kbs = np.asarray(sorted(set(int(k) for k in kbs)))
    cols = np.concatenate([np.arange(kb * 128, (kb + 1) * 128) for kb in kbs])
    q, s = O.quant_weight_128x128(bf16_to_np(w[:, torch.from_numpy(cols)]), pow2)
    return cols, q, s


def assert_gemm_close_whole(c_gpu: torch.Tensor, c_ref: np.ndarray, what: str = "", rows: int = 2048) -> dict:
    """assert_gemm_close over a whole (large) output, compared in row chunks so
    that the temporaries stay small: the same criteria (relative Frobenius
    error, the per-element bound with rms(C_ref) of the whole output, no
    non-finite values) computed over every element."""
    c_ref = np.asarray(c_ref, np.float64)
    rms = float(np.sqrt(np.mean(np.square(c_ref)))) if c_ref.size else 0.0
    ref2 = diff2 = 0.0
    viol = lit = nonfin = 0
    emax = 0.0
    for r0 in range(0, c_ref.shape[0], rows):
        r1 = min(c_ref.shape[0], r0 + rows)
        g = c_gpu[r0:r1].float().cpu().numpy().astype(np.float64)
        ref = c_ref[r0:r1]
        nonfin += int(np.sum(~np.isfinite(g)))
        d = g - ref
        err = np.abs(d)
        diff2 += float(np.sum(np.square(d)))
        ref2 += float(np.sum(np.square(ref)))
        viol += int(np.sum(err > ABS_RMS * rms + BF16_HALF_ULP_REL * np.abs(ref)))
        lit += int(np.sum(err > ABS_RMS * rms))
        if err.size:
            emax = max(emax, float(err.max()))
    e = {"rel_frob": float(np.sqrt(diff2 / ref2)) if ref2 > 0 else float(np.sqrt(diff2)),
         "max_err_over_rms": emax / rms if rms > 0 else 0.0, "violations": viol, "literal_violations": lit,
         "nonfinite": nonfin, "n": int(c_ref.size)}
    assert e["nonfinite"] == 0, (what, e)
    assert e["rel_frob"] <= REL_FROB, (what, e)
    assert e["violations"] == 0, (what, e)
    return e
