"""Every entry of the measured split-K table (csrc/split_table.inc), run with
the K-splits the planner takes from it, against the oracle.

For each entry the call's plan must report the entry's K-splits; C is then
checked on sampled outputs (every activation row at 48 random weight rows,
plus 512 random outputs) against the oracle's dequantize-then-double GEMM of
its own quantization of the same seeded inputs, within 2^-8 * sum|a b| + 1e-3."""
import functools

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_mxfp4_gb300 import workloads as wl
from gpu_util import assert_within_tolerance, dev_bf16, gemm_sampled_parallel

pytestmark = pytest.mark.gpu

mx = pytest.importorskip("block_scaled_fp4_mxfp4_gb300.mxfp4")


@functools.lru_cache(maxsize=40)
def weights(n, k, vec):
    """(bf16 bits, oracle codes and scales, device codes and scales) of a seeded
    weight matrix [n, k], quantized once per shape and format."""
    bits = wl.gen_bf16(11, 3000 + n + k, n, k, "normal", 0.02)
    q_r, sf_r = (oracle.nv_quantize if vec == 16 else oracle.mx_quantize)(bits)
    q, sf = (mx.nvfp4_quantize if vec == 16 else mx.mxfp4_quantize)(dev_bf16(bits))
    return q_r, sf_r, q, sf


def entries():
    try:
        return mx.split_table()
    except Exception:   # no library: the module-level importorskip reports it
        return []


@pytest.mark.parametrize("e", entries(), ids=lambda e: f"{e['path']}-b{e['bucket']}-{e['n']}x{e['k']}-s{e['splits']}")
def test_split_table_entry(e):
    path, n, k = e["path"], e["n"], e["k"]
    nv = path == "fused_nv"
    vec = 16 if nv else 32
    m = e["bucket"] - 3 if path != "gemm" else 128 * e["bucket"] - 5
    plan = mx.gemm_plan(m, n, k, fused=path != "gemm", nvfp4=nv)
    assert plan["splits"] == e["splits"], (plan, e)
    a = wl.gen_bf16(12, m + n + k, m, k)
    q_r, sf_r, qb, sfb = weights(n, k, vec)
    A = dev_bf16(a)
    if path == "gemm":
        aq, asf = mx.mxfp4_quantize(A)
        C = mx.mxfp4_gemm_a4w4(aq, asf, qb, sfb, k)
    elif nv:
        C = mx.nvfp4_quant_gemm_fused(A, qb, sfb)
    else:
        C = mx.mxfp4_quant_gemm_fused(A, qb, sfb)
    torch.cuda.synchronize()
    qa_r, sfa_r = (oracle.nv_quantize if nv else oracle.mx_quantize)(a)
    rng = np.random.default_rng(m * 7 + n + k)
    cols48 = rng.integers(0, n, 48)
    rows = np.concatenate([np.repeat(np.arange(m), 48), rng.integers(0, m, 512)]).astype(np.int64)
    cols = np.concatenate([np.tile(cols48, m), rng.integers(0, n, 512)]).astype(np.int64)
    c_ref, s = gemm_sampled_parallel(qa_r, sfa_r, q_r, sf_r, k, vec, rows, cols)
    got = C[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].double().cpu().numpy()
    assert_within_tolerance(got, c_ref, s, f"{path} {m}x{n}x{k} with {e['splits']} K-splits")
    assert mx.get_device_error() == 0


def test_override_reaches_the_planner_and_clears():
    assert mx.set_split_override("fused", 5) == 0
    try:
        assert mx.gemm_plan(16, 2112, 7168, fused=True)["splits"] == 5
        assert mx.set_split_override("fused", 2) == 5     # below what 8-stage CTAs allow: clamped to 4
        assert mx.gemm_plan(16, 2112, 7168, fused=True)["splits"] == 4
    finally:
        assert mx.set_split_override("fused", 0) == 2
    assert mx.set_split_override("gemm", 4) == 0
    try:
        assert mx.gemm_plan(256, 2112, 4096)["splits"] == 4
    finally:
        mx.set_split_override("gemm", 0)
