"""Helpers for the GPU parity tests: move seeded inputs to the device, run the
CUDA path through the C ABI, run the oracle on the same inputs, compare."""
import numpy as np
import torch

import oracle


def dev_bf16(bits: np.ndarray, pad_cols: int = 0) -> torch.Tensor:
    """bf16 bit patterns -> CUDA bf16 tensor (optionally inside a wider row stride)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    if pad_cols:
        M, K = bits.shape
        big = torch.zeros((M, K + pad_cols), dtype=torch.bfloat16)
        big[:, :K] = t
        return big.cuda()[:, :K]
    return t.cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().cpu().numpy()


def c_f64(C: torch.Tensor) -> np.ndarray:
    return C.float().cpu().numpy().astype(np.float64)


def assert_bytes_equal(got: np.ndarray, want: np.ndarray, what: str):
    got = np.asarray(got).ravel()
    want = np.asarray(want).ravel()
    assert got.shape == want.shape, (what, got.shape, want.shape)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{what}: {bad.size} bytes differ, first at {bad[:8]}: got {got[bad[:8]]} want {want[bad[:8]]}"


def assert_within_tolerance(c_gpu: np.ndarray, c_ref: np.ndarray, s_abs: np.ndarray, what: str):
    """|C_gpu - C_ref| <= 2^-8 * sum_k |a_k b_k| + 1e-3 for every element."""
    bad, worst = oracle.check_tolerance(c_gpu, c_ref, s_abs)
    if bad:
        d = np.abs(np.asarray(c_gpu, np.float64).ravel() - np.asarray(c_ref).ravel())
        bound = np.ldexp(np.asarray(s_abs).ravel(), -8) + 1e-3
        i = np.flatnonzero(~(d <= bound))[:5]
        raise AssertionError(f"{what}: {bad} elements out of tolerance (worst ratio {worst:.3g}); "
                             f"idx {i} gpu {np.asarray(c_gpu).ravel()[i]} ref {np.asarray(c_ref).ravel()[i]}")
    return worst


def gemm_sampled_parallel(qa, sfa, qb, sfb, K: int, vec: int, rows, cols, threads: int = 0):
    """oracle.gemm_sampled over host threads (the oracle's C loop releases the
    GIL; every output is computed by the same definition, so the split changes
    nothing but the wall time)."""
    import concurrent.futures as cf
    import os
    threads = threads or max(1, min(32, len(os.sched_getaffinity(0))))
    n = len(rows)
    edges = [n * i // threads for i in range(threads + 1)]
    parts = [(edges[i], edges[i + 1]) for i in range(threads) if edges[i + 1] > edges[i]]
    with cf.ThreadPoolExecutor(max_workers=len(parts)) as ex:
        res = list(ex.map(lambda lh: oracle.gemm_sampled(qa, sfa, qb, sfb, K, vec, rows[lh[0]:lh[1]],
                                                          cols[lh[0]:lh[1]]), parts))
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])


def sample_pairs(M: int, N: int, n_random: int, n_rows: int, n_cols: int, seed: int):
    """Random (m, n) pairs plus a few full rows and full columns."""
    from block_scaled_fp4_mxfp4_gb300 import workloads as wl
    u = wl.uniform01(wl.stream_key(seed, 99), 2 * n_random + n_rows + n_cols)
    rows = (u[:n_random] * M).astype(np.int64)
    cols = (u[n_random:2 * n_random] * N).astype(np.int64)
    fr = (u[2 * n_random:2 * n_random + n_rows] * M).astype(np.int64)
    fc = (u[2 * n_random + n_rows:] * N).astype(np.int64)
    rows = np.concatenate([rows, np.repeat(fr, N), np.tile(np.arange(M), n_cols)])
    cols = np.concatenate([cols, np.tile(np.arange(N), n_rows), np.repeat(fc, M)])
    return rows, cols
