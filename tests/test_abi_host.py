"""The C-ABI library builds, loads and exports every declared entry point; host
logic (sizes, argument validation) works without a GPU. No compute calls."""
import ctypes

import pytest

from block_scaled_fp4_mxfp4_gb300 import build as libbuild

libbuild.build()
from block_scaled_fp4_mxfp4_gb300 import mxfp4  # noqa: E402

L = mxfp4.lib()


def test_every_declared_symbol_is_exported():
    names = mxfp4.declared_symbols()
    assert len(names) == 27
    for n in names:
        assert hasattr(L, n), n  # ctypes resolves the exported symbol


def test_group_workspace_sizes():
    for f in (L.nvfp4_group_workspace_bytes, L.mxfp4_group_workspace_bytes):
        assert f(1) == 0 and f(16) == 0                      # kernel parameters carry up to 16 problems
        assert f(17) == 17 * 640 and f(256) == 256 * 640     # 4 TMA descriptors + one record per problem
        assert f(0) == 0 and f(-3) == 0 and f((1 << 20) + 1) == 0


def test_wait_limit_setter_returns_previous_and_zero_restores_default():
    default = 2_000_000_000
    assert mxfp4.set_wait_limit_ns(1234) == default
    assert mxfp4.set_wait_limit_ns(0) == 1234
    assert mxfp4.set_wait_limit_ns(0) == default


def test_status_strings_and_version():
    for code, name in mxfp4.STATUS.items():
        assert L.mxfp4_status_string(code).decode() == name
    assert L.mxfp4_status_string(99).decode() == "MXFP4_UNKNOWN_STATUS"
    assert L.mxfp4_abi_version() == 2


@pytest.mark.parametrize("rows,k,vec,want", [
    (16, 7168, 32, 1 * 56 * 512),      # decode A: 224 scale columns -> 56 blocks
    (2112, 7168, 32, 17 * 56 * 512),
    (128, 256, 16, 4 * 512),           # one NVFP4 256-wide K step = 4 blocks
    (130, 96, 32, 2 * 1 * 512),        # ragged rows and columns
    (1, 32, 32, 512),
    (8, 33, 32, 0), (8, 32, 8, 0), (0, 32, 32, 0),
])
def test_sf_bytes(rows, k, vec, want):
    assert L.mxfp4_sf_bytes(rows, k, vec) == want


def test_workspace_bytes_is_a_function_of_shape():
    a = L.mxfp4_workspace_bytes(16, 2112, 7168)
    assert a == L.mxfp4_workspace_bytes(16, 2112, 7168) > 16 * 7168 // 2
    assert L.mxfp4_workspace_bytes(8192, 8192, 8192) >= 8192 * 4096 + 8192 * 256
    assert L.mxfp4_workspace_bytes(16, 2112, 7000) == 0  # K % 32 != 0
    assert L.nvfp4_group_workspace_bytes(8) == 0


def test_quantize_argument_validation_needs_no_gpu():
    q = L.mxfp4_quantize
    assert q(None, 1, 32, 32, 16, 16, 16, None) == 1                 # null A
    assert q(16, 0, 32, 32, 16, 16, 16, None) == 1                   # M = 0
    assert q(16, 1, 48, 48, 16, 32, 16, None) == 2                   # K % 32
    assert q(16, 1, 32, 31, 16, 16, 16, None) == 1                   # lda < K
    assert q(16, 1, 32, 36, 16, 16, 16, None) == 3                   # lda*2 % 16
    assert q(24, 1, 32, 32, 16, 16, 16, None) == 3                   # A misaligned
    assert q(16, 1, 32, 32, 16, 18, 16, None) == 3                   # ldq % 4
    assert L.nvfp4_quantize(16, 1, 40, 40, 16, 32, 16, None) == 2    # K % 16


def test_gemm_argument_validation_needs_no_gpu():
    g = L.mxfp4_gemm_a4w4
    ok = dict(Aq=16, ldaq=16, Asf=16, Bq=16, ldbq=16, Bsf=16, C=16, ldc=8, M=1, N=8, K=32, ws=16,
              wsb=1 << 20, s=None)

    def call(**kw):
        a = dict(ok, **kw)
        return g(a["Aq"], a["ldaq"], a["Asf"], a["Bq"], a["ldbq"], a["Bsf"], a["C"], a["ldc"], a["M"],
                 a["N"], a["K"], a["ws"], a["wsb"], a["s"])

    assert call(C=None) == 1
    assert call(K=48) == 2
    assert call(ldc=4) == 1
    assert call(ldbq=8) == 1
    assert call(ws=None) == 1
    assert call(wsb=0) == 4
    assert call(Bq=8) == 3
    f = L.mxfp4_quant_gemm_fused
    assert f(16, 31, 16, 16, 16, 16, 8, 1, 8, 32, 16, 1 << 20, None) == 1   # lda < K
    assert f(16, 36, 16, 16, 16, 16, 8, 1, 8, 32, 16, 1 << 20, None) == 3   # lda*2 % 16
    assert f(16, 32, 16, 16, 16, 16, 8, 1, 8, 32, 16, 0, None) == 4


def test_group_gemm_validation_needs_no_gpu():
    P = mxfp4.NvProblem
    good = P(64, 128, 256, 16, 16, 16, 16, 16, 128, 128, 128)
    arr = (P * 1)(good)
    assert L.nvfp4_group_gemm(None, 1, None, 0, None) == 1
    assert L.nvfp4_group_gemm(arr, 0, None, 0, None) == 1
    many = (P * 17)(*([good] * 17))
    # more than 16 problems: the device problem table needs a workspace
    assert L.nvfp4_group_gemm(many, 17, None, 0, None) == 1
    assert L.nvfp4_group_gemm(many, 17, 64, 17 * 640 - 1, None) == 4
    assert L.nvfp4_group_gemm(many, 17, 16, 17 * 640, None) == 3     # table needs 64-byte alignment
    assert L.nvfp4_group_gemm(many, (1 << 20) + 1, 64, 1 << 40, None) == 2
    bad_k = (P * 1)(P(64, 128, 250, 16, 16, 16, 16, 16, 128, 128, 128))
    assert L.nvfp4_group_gemm(bad_k, 1, None, 0, None) == 2
    bad_al = (P * 1)(P(64, 128, 256, 24, 16, 16, 16, 16, 128, 128, 128))
    assert L.nvfp4_group_gemm(bad_al, 1, None, 0, None) == 3


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-GPU answer")
def test_valid_call_without_gpu_reports_no_device():
    assert L.mxfp4_quantize(16, 1, 32, 32, 16, 16, 16, None) == 7
    code = ctypes.c_int(-1)
    assert L.mxfp4_get_device_error(ctypes.byref(code)) == 5


def test_plan_argument_validation_needs_no_gpu():
    plan = mxfp4.Plan()
    assert L.mxfp4_gemm_plan(16, 2112, 7168, 1, None) == 1          # no output struct
    assert L.mxfp4_gemm_plan(16, 2112, 7168, 3, ctypes.byref(plan)) == 1   # which must be 0, 1 or 2
    assert L.mxfp4_gemm_plan(65, 2112, 7168, 2, ctypes.byref(plan)) == 2  # fused NVFP4: M <= 64
    assert L.mxfp4_gemm_plan(16, 2112, 7176, 2, ctypes.byref(plan)) == 2  # K % 32 for the fused path too
    assert L.mxfp4_gemm_plan(0, 2112, 7168, 0, ctypes.byref(plan)) == 1
    assert L.mxfp4_gemm_plan(16, 2112, 7000, 0, ctypes.byref(plan)) == 2   # K % 32
    probs = (mxfp4.NvProblem * 1)()
    probs[0] = mxfp4.NvProblem(64, 256, 100, 16, 16, 16, 16, 16, 64, 128, 256)
    assert L.nvfp4_group_gemm_plan(probs, 1, ctypes.byref(plan)) == 2      # K % 16
    assert L.nvfp4_group_gemm_plan(probs, 1, ctypes.byref(plan)) == 2      # (same list, K % 16)


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the no-GPU answer")
def test_plan_without_gpu_reports_no_device():
    plan = mxfp4.Plan()
    assert L.mxfp4_gemm_plan(16, 2112, 7168, 1, ctypes.byref(plan)) == 7


def test_mx_group_gemm_validation_needs_no_gpu():
    P = mxfp4.MxProblem
    good = (P * 1)()
    good[0] = P(64, 256, 512, 16, 16, 16, 16, 16, 256, 256, 256)
    bad_k = (P * 1)()
    bad_k[0] = P(64, 256, 48, 16, 16, 16, 16, 16, 32, 32, 256)      # K % 32
    assert L.mxfp4_group_gemm(bad_k, 1, None, 0, None) == 2
    null = (P * 1)()
    null[0] = P(64, 256, 512, 0, 16, 16, 16, 16, 256, 256, 256)     # null A
    assert L.mxfp4_group_gemm(null, 1, None, 0, None) == 1
    bad_al = (P * 1)()
    bad_al[0] = P(64, 256, 512, 16, 16, 16, 16, 16, 264, 256, 256)  # lda % 16
    assert L.mxfp4_group_gemm(bad_al, 1, None, 0, None) == 3
    many = (P * 20)(*([good[0]] * 20))
    assert L.mxfp4_group_gemm(many, 20, None, 0, None) == 1          # more than 16 need a workspace
    assert L.mxfp4_group_gemm(many, 20, 64, 20 * 640 - 64, None) == 4
    assert L.mxfp4_group_gemm(None, 1, None, 0, None) == 1
    plan = mxfp4.Plan()
    assert L.mxfp4_group_gemm_plan(bad_k, 1, ctypes.byref(plan)) == 2


def test_gemm_ex_argument_validation_needs_no_gpu():
    f = L.mxfp4_gemm_a4w4_ex
    ok = dict(aq=16, ldaq=512, asf=16, bq=16, ldbq=512, bsf=16, c=16, ldc=64, M=8, N=64, K=1024,
              alpha=1.0, beta=0.0, bias=None, ws=16, wsb=1 << 20)
    def call(**kw):
        a = dict(ok, **kw)
        return f(a["aq"], a["ldaq"], a["asf"], a["bq"], a["ldbq"], a["bsf"], a["c"], a["ldc"], a["M"], a["N"],
                 a["K"], a["alpha"], a["beta"], a["bias"], a["ws"], a["wsb"], None)
    assert call(alpha=float("inf")) == 1
    assert call(beta=float("nan")) == 1
    assert call(bias=17) == 3          # bias must be 2-byte aligned
    assert call(K=1000) == 2           # K % 32
    assert call(ws=0) == 1


def test_nvfp4_fused_argument_validation_needs_no_gpu():
    f = L.nvfp4_quant_gemm_fused
    assert f(16, 1024, 16, 512, 16, 16, 64, 65, 64, 1024, None) == 2     # M > 64
    assert f(16, 1024, 16, 512, 16, 16, 64, 8, 64, 1000, None) == 2      # K % 16
    assert f(None, 1024, 16, 512, 16, 16, 64, 8, 64, 1024, None) == 1
    assert f(16, 1028, 16, 512, 16, 16, 64, 8, 64, 1024, None) == 3      # lda * 2 % 16


def test_group_quant_gemm_validation_needs_no_gpu():
    P = mxfp4.NvActProblem
    def one(**kw):
        f = dict(m=64, n=256, k=512, a=16, b=16, sfb=16, c=16, lda=512, ldb=256, ldc=256)
        f.update(kw)
        arr = (P * 1)()
        arr[0] = P(f["m"], f["n"], f["k"], f["a"], f["b"], f["sfb"], f["c"], f["lda"], f["ldb"], f["ldc"])
        return arr
    ws_fn = L.nvfp4_group_quant_gemm_workspace_bytes
    # per group: packed A (64 rows x 256 B) then its blocked E4M3 scales (128 x 32 B), each 256-aligned
    assert ws_fn(one(), 1) == 64 * 256 + 128 * 32
    assert ws_fn(one(m=64, k=7168, lda=7168), 1) == 64 * 3584 + 128 * 448
    two = (P * 2)()
    two[0], two[1] = one()[0], one(m=3, k=48, lda=48)[0]   # 3 x 24 B rows -> 16-byte rows of 32 B
    assert ws_fn(two, 2) == (64 * 256 + 128 * 32) + (256 + 512)
    assert ws_fn(one(k=40, lda=40), 1) == 0                # K % 16
    f = L.nvfp4_group_quant_gemm
    big = 1 << 30
    assert f(one(k=40, lda=40), 1, 16, big, None) == 2
    assert f(one(a=0), 1, 16, big, None) == 1
    assert f(one(lda=500), 1, 16, big, None) == 1          # lda < k
    assert f(one(lda=516), 1, 16, big, None) == 3          # lda * 2 % 16
    assert f(one(a=24), 1, 16, big, None) == 3             # A not 16-byte aligned
    assert f(one(), 1, None, big, None) == 1               # no workspace
    assert f(one(), 1, 24, big, None) == 3                 # workspace alignment
    assert f(one(), 1, 16, 64 * 256, None) == 4            # workspace too small
    seventeen = (P * 17)(*([one()[0]] * 17))
    per = 64 * 256 + 128 * 32
    assert ws_fn(seventeen, 17) == 17 * per + 17 * 640      # + the device problem table
    assert f(seventeen, 17, 64, 17 * per + 17 * 640 - 1, None) == 4
    assert f(None, 1, 16, big, None) == 1


def test_rmsnorm_quantize_validation_needs_no_gpu():
    f = L.mxfp4_rmsnorm_quantize
    ok = dict(X=16, M=4, K=64, ldx=64, w=16, eps=1e-6, Aq=16, ldq=32, sf=16)
    def call(**kw):
        a = dict(ok, **kw)
        return f(a["X"], a["M"], a["K"], a["ldx"], a["w"], a["eps"], a["Aq"], a["ldq"], a["sf"], None)
    assert call(K=48, ldx=48, ldq=24) == 2      # K % 32
    assert call(w=None) == 1
    assert call(eps=-1.0) == 1
    assert call(eps=float("nan")) == 1
    assert call(eps=float("inf")) == 1
    assert call(w=24) == 3                      # weight alignment
    assert call(ldx=68) == 3                    # ldx * 2 % 16
    assert call(X=None) == 1
    g = L.mxfp4_rmsnorm_quantize_ex
    def call_ex(rstd, sumsq, **kw):
        a = dict(ok, **kw)
        return g(a["X"], a["M"], a["K"], a["ldx"], a["w"], a["eps"], a["Aq"], a["ldq"], a["sf"], rstd, sumsq, None)
    assert call_ex(None, None, K=48, ldx=48, ldq=24) == 2
    assert call_ex(18, None) == 3               # rstd 4-byte alignment
    assert call_ex(None, 20) == 3               # sumsq 8-byte alignment
    assert call_ex(None, None, w=None) == 1


def test_split_table_is_well_formed_without_a_gpu():
    """The measured K-split table the planner consults: unique (path, bucket,
    N, K) keys, split counts the kernels accept (1-8 for the fused kernel's
    clusters, 1-16 for the GEMM path), buckets the planner can produce, and
    the sweep's grid fully covered for every path."""
    t = mxfp4.split_table()
    assert len(t) == 160
    keys = {(e["path"], e["bucket"], e["n"], e["k"]) for e in t}
    assert len(keys) == len(t)
    for e in t:
        assert e["path"] in ("gemm", "fused", "fused_nv"), e
        if e["path"] == "gemm":
            assert e["bucket"] in (1, 2) and 1 <= e["splits"] <= 16, e
        else:
            assert e["bucket"] in (16, 32, 64) and 1 <= e["splits"] <= 8, e
        assert e["n"] in (512, 2112, 4096, 7168) and e["k"] in (512, 1024, 2048, 4096, 7168), e
    for path, buckets in (("gemm", (1, 2)), ("fused", (16, 32, 64)), ("fused_nv", (16, 32, 64))):
        got = {(e["bucket"], e["n"], e["k"]) for e in t if e["path"] == path}
        assert got == {(b, n, k) for b in buckets for n in (512, 2112, 4096, 7168) for k in (512, 1024, 2048, 4096, 7168)}
    # every GEMM-path entry keeps one split: the measured best everywhere
    assert all(e["splits"] == 1 for e in t if e["path"] == "gemm")
