"""Python binding of libmxfp4 (the C ABI in include/mxfp4.h).

Argument marshalling only: every function passes device pointers, sizes and the
current CUDA stream to the library entry point of the same name and raises
``Mxfp4Error`` on a non-OK status. All arithmetic runs in the library's CUDA
kernels; there is no fallback. If the library has not been built, importing
this module raises immediately.
"""
import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libmxfp4.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "mxfp4.h")

_i64 = ctypes.c_int64
_p = ctypes.c_void_p
_sz = ctypes.c_size_t
_st = ctypes.c_int

STATUS = {
    0: "MXFP4_OK", 1: "MXFP4_ERR_INVALID_ARG", 2: "MXFP4_ERR_UNSUPPORTED_SHAPE",
    3: "MXFP4_ERR_MISALIGNED", 4: "MXFP4_ERR_WORKSPACE_TOO_SMALL", 5: "MXFP4_ERR_CUDA",
    6: "MXFP4_ERR_DEVICE_TIMEOUT", 7: "MXFP4_ERR_NO_DEVICE",
}
NVFP4_MAX_GROUPS = 16


class Mxfp4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}")
        self.status = status


class NvProblem(ctypes.Structure):
    """nvfp4_problem_t."""
    _fields_ = [("m", _i64), ("n", _i64), ("k", _i64),
                ("a", _p), ("sfa", _p), ("b", _p), ("sfb", _p), ("c", _p),
                ("lda", _i64), ("ldb", _i64), ("ldc", _i64)]


class MxProblem(ctypes.Structure):
    """mxfp4_problem_t (same fields as nvfp4_problem_t)."""
    _fields_ = NvProblem._fields_


class NvActProblem(ctypes.Structure):
    """nvfp4_act_problem_t: a grouped NVFP4 problem with bf16 A."""
    _fields_ = [("m", _i64), ("n", _i64), ("k", _i64),
                ("a", _p), ("b", _p), ("sfb", _p), ("c", _p),
                ("lda", _i64), ("ldb", _i64), ("ldc", _i64)]


class Plan(ctypes.Structure):
    """mxfp4_plan_t: the kernel and tiling a call launches."""
    _fields_ = [("kernel", ctypes.c_int), ("tile_m", ctypes.c_int), ("tile_n", ctypes.c_int),
                ("splits", ctypes.c_int), ("tiles", ctypes.c_int), ("quant_launch", ctypes.c_int)]


KERNEL_NAMES = {1: "fused_quant_gemm_kernel", 2: "bs_gemm_kernel", 3: "bs_gemm_pair_kernel"}


def _load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"libmxfp4.so is not built ({path} missing); run __graft_entry__.build() "
            "or python block_scaled_fp4_mxfp4_gb300/build.py")
    L = ctypes.CDLL(path)
    L.mxfp4_status_string.restype = ctypes.c_char_p
    L.mxfp4_status_string.argtypes = [_st]
    L.mxfp4_abi_version.restype = ctypes.c_int
    L.mxfp4_abi_version.argtypes = []
    L.mxfp4_sf_bytes.restype = _sz
    L.mxfp4_sf_bytes.argtypes = [_i64, _i64, ctypes.c_int]
    L.mxfp4_workspace_bytes.restype = _sz
    L.mxfp4_workspace_bytes.argtypes = [_i64, _i64, _i64]
    L.nvfp4_group_workspace_bytes.restype = _sz
    L.nvfp4_group_workspace_bytes.argtypes = [ctypes.c_int]
    L.mxfp4_group_workspace_bytes.restype = _sz
    L.mxfp4_group_workspace_bytes.argtypes = [ctypes.c_int]
    for name in ("mxfp4_quantize", "nvfp4_quantize"):
        f = getattr(L, name)
        f.restype = _st
        f.argtypes = [_p, _i64, _i64, _i64, _p, _i64, _p, _p]
    L.mxfp4_rmsnorm_quantize.restype = _st
    L.mxfp4_rmsnorm_quantize.argtypes = [_p, _i64, _i64, _i64, _p, ctypes.c_float, _p, _i64, _p, _p]
    L.mxfp4_rmsnorm_quantize_ex.restype = _st
    L.mxfp4_rmsnorm_quantize_ex.argtypes = [_p, _i64, _i64, _i64, _p, ctypes.c_float, _p, _i64, _p, _p, _p, _p]
    L.mxfp4_gemm_a4w4.restype = _st
    L.mxfp4_gemm_a4w4.argtypes = [_p, _i64, _p, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _p, _sz, _p]
    L.mxfp4_gemm_a4w4_ex.restype = _st
    L.mxfp4_gemm_a4w4_ex.argtypes = [_p, _i64, _p, _p, _i64, _p, _p, _i64, _i64, _i64, _i64,
                                     ctypes.c_float, ctypes.c_float, _p, _p, _sz, _p]
    L.mxfp4_quant_gemm_fused.restype = _st
    L.mxfp4_quant_gemm_fused.argtypes = [_p, _i64, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _p, _sz, _p]
    L.nvfp4_quant_gemm_fused.restype = _st
    L.nvfp4_quant_gemm_fused.argtypes = [_p, _i64, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _p]
    L.nvfp4_group_gemm.restype = _st
    L.nvfp4_group_gemm.argtypes = [ctypes.POINTER(NvProblem), ctypes.c_int, _p, _sz, _p]
    L.mxfp4_noalloc_scratch_bytes.restype = _sz
    L.mxfp4_noalloc_scratch_bytes.argtypes = []
    L.mxfp4_gemm_a4w4_noalloc.restype = _st
    L.mxfp4_gemm_a4w4_noalloc.argtypes = [_p, _i64, _p, _p, _i64, _p, _p, _i64, _i64, _i64, _i64, _p]
    L.mxfp4_get_device_error.restype = _st
    L.mxfp4_get_device_error.argtypes = [ctypes.POINTER(ctypes.c_int)]
    L.mxfp4_set_split_override.restype = ctypes.c_int
    L.mxfp4_set_split_override.argtypes = [ctypes.c_int, ctypes.c_int]
    L.mxfp4_split_table_entry.restype = ctypes.c_int
    L.mxfp4_split_table_entry.argtypes = [ctypes.c_int] + [ctypes.c_void_p] * 5
    L.mxfp4_set_wait_limit_ns.restype = ctypes.c_uint64
    L.mxfp4_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.mxfp4_gemm_plan.restype = _st
    L.mxfp4_gemm_plan.argtypes = [_i64, _i64, _i64, ctypes.c_int, ctypes.POINTER(Plan)]
    L.nvfp4_group_gemm_plan.restype = _st
    L.nvfp4_group_gemm_plan.argtypes = [ctypes.POINTER(NvProblem), ctypes.c_int, ctypes.POINTER(Plan)]
    L.nvfp4_group_quant_gemm_workspace_bytes.restype = _sz
    L.nvfp4_group_quant_gemm_workspace_bytes.argtypes = [ctypes.POINTER(NvActProblem), ctypes.c_int]
    L.nvfp4_group_quant_gemm.restype = _st
    L.nvfp4_group_quant_gemm.argtypes = [ctypes.POINTER(NvActProblem), ctypes.c_int, _p, _sz, _p]
    L.mxfp4_group_gemm.restype = _st
    L.mxfp4_group_gemm.argtypes = [ctypes.POINTER(MxProblem), ctypes.c_int, _p, _sz, _p]
    L.mxfp4_group_gemm_plan.restype = _st
    L.mxfp4_group_gemm_plan.argtypes = [ctypes.POINTER(MxProblem), ctypes.c_int, ctypes.POINTER(Plan)]
    return L


_lib = _load()


def lib() -> ctypes.CDLL:
    return _lib


def declared_symbols(header: str = HEADER_PATH):
    """Names of the entry points include/mxfp4.h declares."""
    with open(header) as f:
        text = f.read()
    return re.findall(r"MXFP4_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def _check(status: int, where: str):
    if status != 0:
        raise Mxfp4Error(status, where)


def _stream_ptr(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None, ndim=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")
    if t.dim() == 2 and t.stride(1) != 1:
        raise ValueError(f"{name} must be row-major with unit inner stride")
    return t


# ---------------------------------------------------------------- sizes --

def sf_bytes(rows: int, k: int, vec: int) -> int:
    return int(_lib.mxfp4_sf_bytes(rows, k, vec))


def workspace_bytes(M: int, N: int, K: int) -> int:
    return int(_lib.mxfp4_workspace_bytes(M, N, K))


def new_workspace(M: int, N: int, K: int, device="cuda") -> torch.Tensor:
    """A zero-filled workspace for (M, N, K) (the library keeps it zeroed)."""
    return torch.zeros(max(1, workspace_bytes(M, N, K)), dtype=torch.uint8, device=device)


# --------------------------------------------------------- quantization --

def _quant(fn, vec, A, Aq, A_sf, stream, where):
    _dev(A, "A", torch.bfloat16, 2)
    M, K = A.shape
    if Aq is None:
        # row stride rounded up to 16 bytes so Aq can feed the TMA-based GEMMs
        ld = (K // 2 + 15) // 16 * 16
        Aq = torch.empty((M, ld), dtype=torch.uint8, device=A.device)[:, :K // 2]
    if A_sf is None:
        A_sf = torch.empty(max(1, sf_bytes(M, K, vec)), dtype=torch.uint8, device=A.device)
    _dev(Aq, "Aq", torch.uint8, 2)
    _dev(A_sf, "A_sf", torch.uint8)
    _check(fn(A.data_ptr(), M, K, A.stride(0), Aq.data_ptr(), Aq.stride(0), A_sf.data_ptr(),
              _stream_ptr(stream)), where)
    return Aq, A_sf


def mxfp4_quantize(A, Aq=None, A_sf=None, stream=None):
    """bf16 A [M, K] -> (packed E2M1 [M, K/2] u8, blocked E8M0 scales)."""
    return _quant(_lib.mxfp4_quantize, 32, A, Aq, A_sf, stream, "mxfp4_quantize")


def nvfp4_quantize(A, Aq=None, A_sf=None, stream=None):
    """bf16 A [M, K] -> (packed E2M1 [M, K/2] u8, blocked E4M3 scales)."""
    return _quant(_lib.nvfp4_quantize, 16, A, Aq, A_sf, stream, "nvfp4_quantize")


def mxfp4_rmsnorm_quantize(X, weight, eps: float = 1e-6, Aq=None, A_sf=None, stream=None, stats: bool = False):
    """Fused RMSNorm + MXFP4 quantization: bf16 X [M, K], bf16 weight [K] ->
    (packed E2M1 [M, K/2] u8, blocked E8M0 scales) of the normalized rows.
    With stats=True also returns each row's fp32 reciprocal r [M] and its
    exactly rounded fp64 sum of squares [M]."""
    _dev(X, "X", torch.bfloat16, 2)
    _dev(weight, "weight", torch.bfloat16, 1)
    M, K = X.shape
    if weight.numel() != K or not weight.is_contiguous():
        raise ValueError("weight must be a contiguous [K] bf16 tensor")
    if Aq is None:
        ld = (K // 2 + 15) // 16 * 16
        Aq = torch.empty((M, ld), dtype=torch.uint8, device=X.device)[:, :K // 2]
    if A_sf is None:
        A_sf = torch.empty(max(1, sf_bytes(M, K, 32)), dtype=torch.uint8, device=X.device)
    _dev(Aq, "Aq", torch.uint8, 2)
    _dev(A_sf, "A_sf", torch.uint8)
    if not stats:
        _check(_lib.mxfp4_rmsnorm_quantize(X.data_ptr(), M, K, X.stride(0), weight.data_ptr(), float(eps),
                                           Aq.data_ptr(), Aq.stride(0), A_sf.data_ptr(), _stream_ptr(stream)),
               "mxfp4_rmsnorm_quantize")
        return Aq, A_sf
    rstd = torch.empty(M, dtype=torch.float32, device=X.device)
    sumsq = torch.empty(M, dtype=torch.float64, device=X.device)
    _check(_lib.mxfp4_rmsnorm_quantize_ex(X.data_ptr(), M, K, X.stride(0), weight.data_ptr(), float(eps),
                                          Aq.data_ptr(), Aq.stride(0), A_sf.data_ptr(), rstd.data_ptr(),
                                          sumsq.data_ptr(), _stream_ptr(stream)),
           "mxfp4_rmsnorm_quantize_ex")
    return Aq, A_sf, rstd, sumsq


# ------------------------------------------------------------------ GEMM --

def mxfp4_gemm_a4w4(Aq, A_sf, Bq, B_sf, K: int, C=None, workspace=None, stream=None):
    """C [M, N] bf16 = (Aq, A_sf) x (Bq, B_sf)^T."""
    _dev(Aq, "Aq", torch.uint8, 2)
    _dev(Bq, "Bq", torch.uint8, 2)
    M, N = Aq.shape[0], Bq.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=Aq.device)
    if workspace is None:
        workspace = new_workspace(M, N, K, Aq.device)
    _dev(C, "C", torch.bfloat16, 2)
    _check(_lib.mxfp4_gemm_a4w4(Aq.data_ptr(), Aq.stride(0), A_sf.data_ptr(), Bq.data_ptr(),
                                Bq.stride(0), B_sf.data_ptr(), C.data_ptr(), C.stride(0), M, N, K,
                                workspace.data_ptr(), workspace.numel(), _stream_ptr(stream)),
           "mxfp4_gemm_a4w4")
    return C


def mxfp4_gemm_a4w4_ex(Aq, A_sf, Bq, B_sf, K: int, C=None, alpha: float = 1.0, beta: float = 0.0,
                       bias=None, workspace=None, stream=None):
    """C = bf16(alpha * (A_q . B_q^T) + beta * C + bias[n]) (see include/mxfp4.h)."""
    _dev(Aq, "Aq", torch.uint8, 2)
    _dev(Bq, "Bq", torch.uint8, 2)
    M, N = Aq.shape[0], Bq.shape[0]
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs the input C")
        C = torch.empty((M, N), dtype=torch.bfloat16, device=Aq.device)
    _dev(C, "C", torch.bfloat16, 2)
    if bias is not None:
        _dev(bias, "bias", torch.bfloat16, 1)
        if bias.numel() != N:
            raise ValueError(f"bias must have N = {N} elements")
    if workspace is None:
        workspace = new_workspace(M, N, K, Aq.device)
    _check(_lib.mxfp4_gemm_a4w4_ex(Aq.data_ptr(), Aq.stride(0), A_sf.data_ptr(), Bq.data_ptr(), Bq.stride(0),
                                   B_sf.data_ptr(), C.data_ptr(), C.stride(0), M, N, K, float(alpha), float(beta),
                                   bias.data_ptr() if bias is not None else None, workspace.data_ptr(),
                                   workspace.numel(), _stream_ptr(stream)),
           "mxfp4_gemm_a4w4_ex")
    return C


def mxfp4_gemm_a4w4_noalloc(Aq, A_sf, Bq, B_sf, K: int, C, stream=None):
    """The MXFP4 GEMM with the library's fixed scratch array instead of a workspace,
    for callers that cannot allocate device memory (C must be given)."""
    _dev(Aq, "Aq", torch.uint8, 2)
    _dev(Bq, "Bq", torch.uint8, 2)
    _dev(C, "C", torch.bfloat16, 2)
    M, N = Aq.shape[0], Bq.shape[0]
    _check(_lib.mxfp4_gemm_a4w4_noalloc(Aq.data_ptr(), Aq.stride(0), A_sf.data_ptr(), Bq.data_ptr(),
                                        Bq.stride(0), B_sf.data_ptr(), C.data_ptr(), C.stride(0), M, N, K,
                                        _stream_ptr(stream)),
           "mxfp4_gemm_a4w4_noalloc")
    return C


def mxfp4_quant_gemm_fused(A, Bq, B_sf, C=None, workspace=None, stream=None):
    """C [M, N] bf16 = MXFP4(A) x (Bq, B_sf)^T, quantization fused into the GEMM."""
    _dev(A, "A", torch.bfloat16, 2)
    _dev(Bq, "Bq", torch.uint8, 2)
    M, K = A.shape
    N = Bq.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    if workspace is None:
        workspace = new_workspace(M, N, K, A.device)
    _dev(C, "C", torch.bfloat16, 2)
    _check(_lib.mxfp4_quant_gemm_fused(A.data_ptr(), A.stride(0), Bq.data_ptr(), Bq.stride(0),
                                       B_sf.data_ptr(), C.data_ptr(), C.stride(0), M, N, K,
                                       workspace.data_ptr(), workspace.numel(), _stream_ptr(stream)),
           "mxfp4_quant_gemm_fused")
    return C


def nvfp4_quant_gemm_fused(A, Bq, B_sf, C=None, stream=None):
    """C [M, N] fp16 = NVFP4(A) x (Bq, B_sf)^T for M <= 64, quantization fused into the GEMM."""
    _dev(A, "A", torch.bfloat16, 2)
    _dev(Bq, "Bq", torch.uint8, 2)
    M, K = A.shape
    N = Bq.shape[0]
    if C is None:
        C = torch.empty((M, N), dtype=torch.float16, device=A.device)
    _dev(C, "C", torch.float16, 2)
    _check(_lib.nvfp4_quant_gemm_fused(A.data_ptr(), A.stride(0), Bq.data_ptr(), Bq.stride(0), B_sf.data_ptr(),
                                       C.data_ptr(), C.stride(0), M, N, K, _stream_ptr(stream)),
           "nvfp4_quant_gemm_fused")
    return C


def make_nv_problems(groups, struct=None):
    """ctypes array of nvfp4_problem_t (or `struct`) from dicts with keys a, sfa,
    b, sfb, c, k."""
    struct = struct or NvProblem
    arr = (struct * len(groups))()
    for i, g in enumerate(groups):
        a, b, c = g["a"], g["b"], g["c"]
        for name, t in (("a", a), ("b", b), ("c", c), ("sfa", g["sfa"]), ("sfb", g["sfb"])):
            _dev(t, name)
        arr[i] = struct(a.shape[0], b.shape[0], g["k"], a.data_ptr(), g["sfa"].data_ptr(),
                           b.data_ptr(), g["sfb"].data_ptr(), c.data_ptr(),
                           a.stride(0), b.stride(0), c.stride(0))
    return arr


def make_mx_problems(groups):
    """ctypes array of mxfp4_problem_t from dicts with keys a, sfa, b, sfb, c, k."""
    return make_nv_problems(groups, MxProblem)


def group_workspace(num_groups: int, device="cuda", nvfp4: bool = True):
    """Workspace for a grouped GEMM of num_groups problems (None when none is
    needed: up to 16 problems travel in kernel parameters)."""
    n = int((_lib.nvfp4_group_workspace_bytes if nvfp4 else _lib.mxfp4_group_workspace_bytes)(num_groups))
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def _ws_args(workspace):
    return (workspace.data_ptr(), workspace.numel()) if workspace is not None else (None, 0)


def mxfp4_group_gemm(groups, problems=None, workspace=None, stream=None):
    """Grouped MXFP4 GEMM (bf16 C) over `groups` (see make_mx_problems); returns the C list."""
    if problems is None:
        problems = make_mx_problems(groups)
    if workspace is None and len(problems) > NVFP4_MAX_GROUPS:
        workspace = group_workspace(len(problems), groups[0]["c"].device, nvfp4=False)
    _check(_lib.mxfp4_group_gemm(problems, len(problems), *_ws_args(workspace), _stream_ptr(stream)),
           "mxfp4_group_gemm")
    return [g["c"] for g in groups]


def mxfp4_group_gemm_plan(problems) -> dict:
    """What mxfp4_group_gemm launches for these problems (see make_mx_problems)."""
    p = Plan()
    _check(lib().mxfp4_group_gemm_plan(problems, len(problems), ctypes.byref(p)), "mxfp4_group_gemm_plan")
    return _plan_dict(p)


def nvfp4_group_gemm(groups, problems=None, workspace=None, stream=None):
    """Grouped NVFP4 GEMM over `groups` (see make_nv_problems); returns the C list."""
    if problems is None:
        problems = make_nv_problems(groups)
    if workspace is None and len(problems) > NVFP4_MAX_GROUPS:
        workspace = group_workspace(len(problems), groups[0]["c"].device)
    _check(_lib.nvfp4_group_gemm(problems, len(problems), *_ws_args(workspace), _stream_ptr(stream)),
           "nvfp4_group_gemm")
    return [g["c"] for g in groups]


def make_nv_act_problems(groups):
    """ctypes array of nvfp4_act_problem_t from dicts with keys a (bf16 [m, k]),
    b, sfb, c."""
    arr = (NvActProblem * len(groups))()
    for i, g in enumerate(groups):
        a, b, c = g["a"], g["b"], g["c"]
        _dev(a, "a", torch.bfloat16, 2)
        for name, t in (("b", b), ("c", c), ("sfb", g["sfb"])):
            _dev(t, name)
        arr[i] = NvActProblem(a.shape[0], b.shape[0], a.shape[1], a.data_ptr(), b.data_ptr(),
                              g["sfb"].data_ptr(), c.data_ptr(), a.stride(0), b.stride(0), c.stride(0))
    return arr


def nvfp4_group_quant_gemm_workspace_bytes(problems) -> int:
    return int(_lib.nvfp4_group_quant_gemm_workspace_bytes(problems, len(problems)))


def nvfp4_group_quant_gemm(groups, problems=None, workspace=None, stream=None):
    """Grouped NVFP4 GEMM from bf16 activations (quantized in the call) over
    `groups` (see make_nv_act_problems); returns the C list."""
    if problems is None:
        problems = make_nv_act_problems(groups)
    if workspace is None:
        n = nvfp4_group_quant_gemm_workspace_bytes(problems)
        workspace = torch.empty(max(1, n), dtype=torch.uint8, device=groups[0]["a"].device)
    _check(_lib.nvfp4_group_quant_gemm(problems, len(problems), workspace.data_ptr(), workspace.numel(),
                                       _stream_ptr(stream)), "nvfp4_group_quant_gemm")
    return [g["c"] for g in groups]


def _plan_dict(p: Plan) -> dict:
    return dict(kernel=KERNEL_NAMES.get(p.kernel, str(p.kernel)), tile_m=p.tile_m, tile_n=p.tile_n,
                splits=p.splits, tiles=p.tiles, quant_launch=bool(p.quant_launch))


def gemm_plan(M: int, N: int, K: int, fused: bool = False, nvfp4: bool = False) -> dict:
    """What mxfp4_gemm_a4w4 (fused=False), mxfp4_quant_gemm_fused (fused=True) or
    nvfp4_quant_gemm_fused (nvfp4=True) launches for an M x N x K problem on the
    current device."""
    p = Plan()
    which = 2 if nvfp4 else (1 if fused else 0)
    _check(lib().mxfp4_gemm_plan(M, N, K, which, ctypes.byref(p)), "mxfp4_gemm_plan")
    return _plan_dict(p)


def nvfp4_group_gemm_plan(problems) -> dict:
    """What nvfp4_group_gemm launches for these problems (see make_nv_problems)."""
    p = Plan()
    _check(lib().nvfp4_group_gemm_plan(problems, len(problems), ctypes.byref(p)), "nvfp4_group_gemm_plan")
    return _plan_dict(p)


SPLIT_PATHS = {"gemm": 0, "fused": 1, "fused_nv": 2}


def set_split_override(path: str, splits: int) -> int:
    """Override the K-splits of later calls on `path` ("gemm", "fused",
    "fused_nv"; 0 clears); returns the previous override."""
    r = int(_lib.mxfp4_set_split_override(SPLIT_PATHS[path], int(splits)))
    if r < 0:
        raise ValueError("bad split override")
    return r


def split_table():
    """The measured split-K table built into the library: a list of dicts
    (path, bucket, n, k, splits)."""
    names = {v: k for k, v in SPLIT_PATHS.items()}
    n = int(_lib.mxfp4_split_table_entry(-1, None, None, None, None, None))
    out = []
    for i in range(n):
        path, bucket, splits = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        nn, kk = ctypes.c_int64(), ctypes.c_int64()
        _lib.mxfp4_split_table_entry(i, ctypes.byref(path), ctypes.byref(bucket), ctypes.byref(nn),
                                     ctypes.byref(kk), ctypes.byref(splits))
        out.append(dict(path=names[path.value], bucket=bucket.value, n=nn.value, k=kk.value, splits=splits.value))
    return out


def set_wait_limit_ns(ns: int) -> int:
    """Limit of the kernels' work-guarding waits for later launches (0: the
    default of 2 s); returns the previous limit."""
    return int(_lib.mxfp4_set_wait_limit_ns(int(ns)))


def get_device_error() -> int:
    code = ctypes.c_int(0)
    _check(_lib.mxfp4_get_device_error(ctypes.byref(code)), "mxfp4_get_device_error")
    return code.value
