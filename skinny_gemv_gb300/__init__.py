"""Python binding of the GB300 bf16 GEMM / skinny-GEMV C library.

Argument marshalling only: every function here forwards device pointers, sizes
and the current CUDA stream to ``libskinny_gemm.so`` through ctypes; all of C is
computed by the library's sm_103a kernels.  PyTorch is used for device memory
and streams.  If the library has not been built the import of any compute
function raises -- there is no fallback.

    import torch, skinny_gemv_gb300 as sg
    C = sg.gemm_bf16(A, B)        # A [M, K], B [N, K] bf16 on cuda -> C [M, N] = A @ B.T
    C = sg.gemv_bf16(x, W)        # x [M <= 64, K]
"""
from __future__ import annotations

import ctypes
import os
import re

from . import _build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "skinny_gemm.h")

SG_OK = 0
SG_ERR_INVALID_ARG = 1
SG_ERR_MISALIGNED = 2
SG_ERR_UNSUPPORTED_DEVICE = 3
SG_ERR_CUDA = 4
SG_ERR_TIMEOUT = 5
SG_ERR_OUT_OF_MEMORY = 6

PATH_AUTO = 0
PATH_CUDA_CORE = 1
PATH_TENSOR_CORE = 2
PATH_GEMM = 3
PATH_GEMM_PAIR = 4
PATH_NAMES = {PATH_AUTO: "auto", PATH_CUDA_CORE: "cuda_core", PATH_TENSOR_CORE: "tensor_core",
              PATH_GEMM: "gemm", PATH_GEMM_PAIR: "gemm_pair"}


class SgError(RuntimeError):
    def __init__(self, status: int, where: str, lib=None):
        self.status = status
        msg = lib.sg_status_string(status).decode() if lib is not None else f"status {status}"
        if status == SG_ERR_CUDA and lib is not None:
            msg += f" (cudaError {lib.sg_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")


class PlanInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
                ("tile_k", ctypes.c_int32), ("tiles_m", ctypes.c_int32), ("tiles_n", ctypes.c_int32),
                ("k_steps", ctypes.c_int32), ("grid", ctypes.c_int32), ("dp_tiles", ctypes.c_int32),
                ("sk_tiles", ctypes.c_int32), ("sk_units", ctypes.c_int64), ("group_m", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("split_k", ctypes.c_int32), ("rows_per_cta", ctypes.c_int32),
                ("wave_efficiency", ctypes.c_double), ("cluster_size", ctypes.c_int32),
                ("ctas_per_sm", ctypes.c_int32), ("prefetch_steps", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


class DeviceInfo(ctypes.Structure):
    _fields_ = [("sm_count", ctypes.c_int32), ("cc_major", ctypes.c_int32), ("cc_minor", ctypes.c_int32),
                ("smem_optin_bytes", ctypes.c_int32), ("l2_bytes", ctypes.c_int32),
                ("global_mem_bytes", ctypes.c_int64), ("clock_khz", ctypes.c_int32),
                ("mem_clock_khz", ctypes.c_int32), ("mem_bus_bits", ctypes.c_int32)]


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False):
    """The loaded ctypes library.  Raises if it is not built (no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB_PATH):
        if not build_if_missing:
            raise RuntimeError(f"CUDA library not built: {_build.LIB_PATH} is missing; "
                               "run __graft_entry__.build() (nvcc, sm_103a)")
        _build.build()
    lib = ctypes.CDLL(_build.LIB_PATH)
    p, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    for name in ("gemm_bf16", "gemv_bf16", "gemv_bf16_noalloc"):
        f = getattr(lib, name)
        f.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64, p]
        f.restype = ctypes.c_int
    for name in ("gemv_bf16_path", "gemm_bf16_path"):
        f = getattr(lib, name)
        f.argtypes = [p, p, p, i64, i64, i64, i64, i64, i64, ctypes.c_int, p]
        f.restype = ctypes.c_int
    lib.gemm_bf16_swiglu.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, i64, p]
    lib.gemm_bf16_swiglu.restype = ctypes.c_int
    lib.gemm_bf16_swiglu_path.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, i64, ctypes.c_int, p]
    lib.gemm_bf16_swiglu_path.restype = ctypes.c_int
    lib.gemm_bf16_residual.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, i64, i64, p]
    lib.gemm_bf16_residual.restype = ctypes.c_int
    lib.gemm_bf16_residual_path.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, i64, i64, ctypes.c_int, p]
    lib.gemm_bf16_residual_path.restype = ctypes.c_int
    pp, p64 = ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_int64)
    lib.gemv_bf16_batched.argtypes = [p, i64, i64, i64, pp, p64, p64, pp, p64, ctypes.c_int, ctypes.c_int, p]
    lib.gemv_bf16_batched.restype = ctypes.c_int
    lib.gemm_nvfp4.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, i64, ctypes.c_float, p]
    lib.gemm_nvfp4.restype = ctypes.c_int
    lib.nvfp4_scale_bytes.argtypes = [i64, i64]
    lib.nvfp4_scale_bytes.restype = i64
    lib.nvfp4_pack_scales.argtypes = [p, i64, i64, i64, p, p]
    lib.nvfp4_pack_scales.restype = ctypes.c_int
    lib.sg_plan_nvfp4.argtypes = [i64, i64, i64, i32, i32, ctypes.POINTER(PlanInfo)]
    lib.gemm_nvfp4_path.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, i64, ctypes.c_float, ctypes.c_int, p]
    lib.gemm_nvfp4_path.restype = ctypes.c_int
    lib.attention_bf16.argtypes = [p, p, p, p] + [i64] * 10 + [ctypes.c_int, ctypes.c_float, p]
    lib.attention_bf16.restype = ctypes.c_int
    lib.attention_bf16_path.argtypes = [p, p, p, p] + [i64] * 10 + [ctypes.c_int, ctypes.c_float, ctypes.c_int, p]
    lib.attention_bf16_path.restype = ctypes.c_int
    lib.sg_plan_nvfp4.restype = ctypes.c_int
    lib.sg_status_string.argtypes = [ctypes.c_int]
    lib.sg_status_string.restype = ctypes.c_char_p
    lib.sg_last_cuda_error.argtypes = []
    lib.sg_last_cuda_error.restype = ctypes.c_int
    lib.sg_check_device_errors.argtypes = [p, ctypes.POINTER(ctypes.c_uint32)]
    lib.sg_check_device_errors.restype = ctypes.c_int
    lib.sg_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.sg_set_wait_timeout_ns.restype = None
    lib.sg_debug_inject_missing_tx.argtypes = [ctypes.c_uint32]
    lib.sg_debug_inject_missing_tx.restype = None
    lib.sg_plan.argtypes = [i64, i64, i64, i32, i32, ctypes.POINTER(PlanInfo)]
    lib.sg_plan.restype = ctypes.c_int
    lib.sg_plan_swiglu.argtypes = [i64, i64, i64, i32, i32, ctypes.POINTER(PlanInfo)]
    lib.sg_plan_swiglu.restype = ctypes.c_int
    lib.sg_plan_item.argtypes = [ctypes.POINTER(PlanInfo), i32, i32, ctypes.POINTER(ctypes.c_int32)]
    lib.sg_plan_item.restype = ctypes.c_int
    lib.sg_wave_efficiency.argtypes = [i64, i64]
    lib.sg_wave_efficiency.restype = ctypes.c_double
    lib.sg_device_query.argtypes = [ctypes.POINTER(DeviceInfo)]
    lib.sg_device_query.restype = ctypes.c_int
    dp = ctypes.POINTER(ctypes.c_double)
    lib.sg_bench_tcgen05_peak.argtypes = [i64, dp, dp, p]
    lib.sg_bench_tcgen05_peak.restype = ctypes.c_int
    lib.sg_bench_copy.argtypes = [p, p, i64, i32, dp, p]
    lib.sg_bench_copy.restype = ctypes.c_int
    lib.sg_bench_read.argtypes = [p, i64, i32, p, dp, p]
    lib.sg_bench_read.restype = ctypes.c_int
    _lib = lib
    return lib


def declared_symbols() -> list[str]:
    """Function names declared in include/skinny_gemm.h."""
    text = open(HEADER).read()
    return re.findall(r"^SG_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)


def _check(status: int, where: str) -> None:
    if status != SG_OK:
        raise SgError(status, where, load())


# ------------------------------------------------------------------ raw pointers
def gemm_bf16_ptr(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                  stream: int = 0, path: int = PATH_AUTO) -> int:
    """C-ABI call with raw device pointers; returns the sg_status code."""
    return load().gemm_bf16_path(A, B, C, M, N, K, lda, ldb, ldc, path, stream)


def gemv_bf16_ptr(A: int, B: int, C: int, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                  stream: int = 0, path: int = PATH_AUTO) -> int:
    return load().gemv_bf16_path(A, B, C, M, N, K, lda, ldb, ldc, path, stream)


# ------------------------------------------------------------------ torch tensors
def _torch():
    import torch
    return torch


def _operand(t, name: str):
    torch = _torch()
    if t.dtype != torch.bfloat16 or t.dim() != 2 or not t.is_cuda:
        raise ValueError(f"{name} must be a 2-D bfloat16 CUDA tensor, got {t.dtype} {tuple(t.shape)} {t.device}")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit stride along its last dimension")
    return t.data_ptr(), max(t.stride(0), t.shape[1])


def _stream_handle(stream) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _call(fn_name: str, A, B, C=None, stream=None, path: int | None = None):
    torch = _torch()
    a_ptr, lda = _operand(A, "A")
    b_ptr, ldb = _operand(B, "B")
    M, K = A.shape
    N, Kb = B.shape
    if Kb != K:
        raise ValueError(f"K mismatch: A is {tuple(A.shape)}, B is {tuple(B.shape)}")
    if C is None:
        ld = -(-N // 8) * 8  # rows 16-byte aligned, as the library requires
        C = torch.empty((M, ld), dtype=torch.bfloat16, device=A.device)[:, :N]
    c_ptr, ldc = _operand(C, "C")
    if tuple(C.shape) != (M, N):
        raise ValueError(f"C must be {(M, N)}, got {tuple(C.shape)}")
    s = _stream_handle(stream)
    lib = load()
    with torch.cuda.device(A.device):
        if fn_name == "gemm_bf16":
            st = lib.gemm_bf16_path(a_ptr, b_ptr, c_ptr, M, N, K, lda, ldb, ldc,
                                    PATH_AUTO if path is None else path, s)
        elif fn_name == "gemv_bf16_noalloc":
            st = lib.gemv_bf16_noalloc(a_ptr, b_ptr, c_ptr, M, N, K, lda, ldb, ldc, s)
        else:
            st = lib.gemv_bf16_path(a_ptr, b_ptr, c_ptr, M, N, K, lda, ldb, ldc,
                                    PATH_AUTO if path is None else path, s)
    _check(st, fn_name)
    return C


def gemm_bf16(A, B, C=None, stream=None, path: int = PATH_AUTO):
    """C[M, N] = A[M, K] @ B[N, K]^T in bf16 with fp32 accumulation; ``path``
    picks the kernel (PATH_AUTO, PATH_GEMM, PATH_GEMM_PAIR, or a skinny PATH_*)."""
    return _call("gemm_bf16", A, B, C, stream, path)


def gemm_bf16_swiglu(A, Wg, Wu, C=None, stream=None, path: int = PATH_AUTO):
    """C[M, N] = silu(A @ Wg^T) * (A @ Wu^T) in one launch (fp32 accumulation and
    epilogue, bf16 out); Wg and Wu are [N, K] with one leading dimension."""
    torch = _torch()
    a_ptr, lda = _operand(A, "A")
    g_ptr, ldg = _operand(Wg, "Wg")
    u_ptr, ldu = _operand(Wu, "Wu")
    M, K = A.shape
    N = Wg.shape[0]
    if tuple(Wg.shape) != (N, K) or tuple(Wu.shape) != (N, K):
        raise ValueError(f"Wg and Wu must both be {(N, K)}: {tuple(Wg.shape)} {tuple(Wu.shape)}")
    if ldg != ldu:
        raise ValueError(f"Wg and Wu must share a leading dimension ({ldg} vs {ldu})")
    if C is None:
        ld = -(-N // 8) * 8
        C = torch.empty((M, ld), dtype=torch.bfloat16, device=A.device)[:, :N]
    c_ptr, ldc = _operand(C, "C")
    if tuple(C.shape) != (M, N):
        raise ValueError(f"C must be {(M, N)}, got {tuple(C.shape)}")
    with torch.cuda.device(A.device):
        st = load().gemm_bf16_swiglu_path(a_ptr, g_ptr, u_ptr, c_ptr, M, N, K, lda, ldg, ldc, path,
                                          _stream_handle(stream))
    _check(st, "gemm_bf16_swiglu")
    return C


def gemm_bf16_residual(A, B, R, C=None, stream=None, path: int = PATH_AUTO):
    """C[M, N] = A @ B^T + R with the sum in fp32 and one bf16 rounding; R may be C
    (in place)."""
    torch = _torch()
    a_ptr, lda = _operand(A, "A")
    b_ptr, ldb = _operand(B, "B")
    r_ptr, ldr = _operand(R, "R")
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K or tuple(R.shape) != (M, N):
        raise ValueError(f"shapes: A {tuple(A.shape)}, B {tuple(B.shape)}, R {tuple(R.shape)}")
    if C is None:
        ld = -(-N // 8) * 8
        C = torch.empty((M, ld), dtype=torch.bfloat16, device=A.device)[:, :N]
    c_ptr, ldc = _operand(C, "C")
    if tuple(C.shape) != (M, N):
        raise ValueError(f"C must be {(M, N)}, got {tuple(C.shape)}")
    with torch.cuda.device(A.device):
        st = load().gemm_bf16_residual_path(a_ptr, b_ptr, r_ptr, c_ptr, M, N, K, lda, ldb, ldr, ldc, path,
                                            _stream_handle(stream))
    _check(st, "gemm_bf16_residual")
    return C


def _bytes_operand(t, name: str):
    torch = _torch()
    if t.dtype != torch.uint8 or t.dim() != 2 or not t.is_cuda:
        raise ValueError(f"{name} must be a 2-D uint8 CUDA tensor, got {t.dtype} {tuple(t.shape)} {t.device}")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit stride along its last dimension")
    return t.data_ptr(), max(t.stride(0), t.shape[1])


def nvfp4_scale_bytes(rows: int, K: int) -> int:
    """Bytes of the scale-atom buffer gemm_nvfp4 reads for `rows` rows."""
    return int(load().nvfp4_scale_bytes(rows, K))


def nvfp4_pack_scales(plain, K: int | None = None, atoms=None, stream=None):
    """Plain row-major E4M3 scale codes (uint8 [rows, >= K/16]) to the scale atoms
    gemm_nvfp4 reads (a flat uint8 tensor); padding is written as 0."""
    torch = _torch()
    p_ptr, ld = _bytes_operand(plain, "plain")
    rows = plain.shape[0]
    K = 16 * plain.shape[1] if K is None else K
    n = nvfp4_scale_bytes(rows, K)
    if atoms is None:
        atoms = torch.empty(max(n, 1), dtype=torch.uint8, device=plain.device)
    if atoms.dtype != torch.uint8 or not atoms.is_cuda or atoms.numel() < n or not atoms.is_contiguous():
        raise ValueError(f"atoms must be a contiguous uint8 CUDA tensor of at least {n} bytes")
    with torch.cuda.device(plain.device):
        st = load().nvfp4_pack_scales(p_ptr, rows, K, ld, atoms.data_ptr(), _stream_handle(stream))
    _check(st, "nvfp4_pack_scales")
    return atoms


def gemm_nvfp4(A, SFA, B, SFB, K: int | None = None, C=None, alpha: float = 1.0, stream=None,
               path: int = PATH_AUTO):
    """C[M, N] (fp16) = alpha * (A . SFA) @ (B . SFB)^T for packed E2M1 operands
    (uint8 [M, >= K/2] and [N, >= K/2]) and their E4M3 scale atoms (from
    nvfp4_pack_scales)."""
    torch = _torch()
    a_ptr, lda = _bytes_operand(A, "A")
    b_ptr, ldb = _bytes_operand(B, "B")
    M, N = A.shape[0], B.shape[0]
    K = 2 * A.shape[1] if K is None else K
    if 2 * A.shape[1] < K or 2 * B.shape[1] < K:
        raise ValueError(f"K = {K} needs {K // 2} bytes per row: A {tuple(A.shape)}, B {tuple(B.shape)}")
    for t, rows, name in ((SFA, M, "SFA"), (SFB, N, "SFB")):
        if t.dtype != torch.uint8 or not t.is_cuda or t.numel() < nvfp4_scale_bytes(rows, K):
            raise ValueError(f"{name} must hold nvfp4_scale_bytes({rows}, {K}) uint8 scale-atom bytes")
    if C is None:
        ld = -(-N // 8) * 8
        C = torch.empty((M, ld), dtype=torch.float16, device=A.device)[:, :N]
    if C.dtype != torch.float16 or tuple(C.shape) != (M, N) or not C.is_cuda or (N > 1 and C.stride(1) != 1):
        raise ValueError(f"C must be a float16 CUDA tensor of shape {(M, N)}")
    ldc = max(C.stride(0), N)
    with torch.cuda.device(A.device):
        st = load().gemm_nvfp4_path(a_ptr, SFA.data_ptr(), b_ptr, SFB.data_ptr(), C.data_ptr(), M, N, K, lda, ldb,
                                    ldc, float(alpha), int(path), _stream_handle(stream))
    _check(st, "gemm_nvfp4_path")
    return C


def _tokens_heads(t, name: str):
    """A [B, S, heads, D] bfloat16 CUDA tensor whose (heads, D) block is dense:
    returns (pointer, token pitch in elements)."""
    torch = _torch()
    if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_cuda:
        raise ValueError(f"{name} must be a 4-D [batch, seq, heads, head_dim] bfloat16 CUDA tensor, "
                         f"got {t.dtype} {tuple(t.shape)} {t.device}")
    Bt, S, H, D = t.shape
    if (D > 1 and t.stride(3) != 1) or (H > 1 and t.stride(2) != D):
        raise ValueError(f"{name} must have dense heads x head_dim rows")
    # token row b * S + i at pitch ld; with one token per sequence the rows are
    # the batches (a size-1 dimension's stride says nothing about memory)
    if S > 1:
        ld = t.stride(1)
        if Bt > 1 and t.stride(0) != S * ld:
            raise ValueError(f"{name} must have batches of whole rows")
    elif Bt > 1:
        ld = t.stride(0)
    else:
        ld = H * D
    if ld < H * D:  # overlapping or broadcast rows: not a token-major layout
        raise ValueError(f"{name} token rows overlap (pitch {ld} < {H * D} elements)")
    return t.data_ptr(), ld


def attention_bf16(Q, K, V, O=None, causal: bool = False, scale: float | None = None, stream=None,
                   path: int = PATH_AUTO):
    """O = softmax(scale Q K^T, causal mask) V per head for Q [B, Sq, H, 128] and
    K, V [B, Sk, Hkv, 128] (bfloat16); returns O [B, Sq, H, 128].  ``path``:
    PATH_AUTO, PATH_TENSOR_CORE (the tcgen05 kernel) or PATH_CUDA_CORE (the
    decode kernel, Sq x H / Hkv <= 4)."""
    torch = _torch()
    q_ptr, ldq = _tokens_heads(Q, "Q")
    k_ptr, ldk = _tokens_heads(K, "K")
    v_ptr, ldv = _tokens_heads(V, "V")
    Bt, Sq, H, D = Q.shape
    Sk, Hkv = K.shape[1], K.shape[2]
    if tuple(K.shape) != (Bt, Sk, Hkv, D) or tuple(V.shape) != tuple(K.shape):
        raise ValueError(f"K and V must be [{Bt}, seq_k, kv_heads, {D}], got {tuple(K.shape)} and {tuple(V.shape)}")
    if O is None:
        O = torch.empty((Bt, Sq, H, D), dtype=torch.bfloat16, device=Q.device)
    if tuple(O.shape) != (Bt, Sq, H, D):
        raise ValueError(f"O must be [{Bt}, {Sq}, {H}, {D}]")
    o_ptr, ldo = _tokens_heads(O, "O")
    scale = D ** -0.5 if scale is None else float(scale)
    with torch.cuda.device(Q.device):
        st = load().attention_bf16_path(q_ptr, k_ptr, v_ptr, o_ptr, Bt, Sq, Sk, H, Hkv, D, ldq, ldk, ldv, ldo,
                                        1 if causal else 0, scale, path, _stream_handle(stream))
    _check(st, "attention_bf16_path")
    return O


def gemv_bf16_batched(A, Bs, Cs=None, stream=None, path: int = PATH_AUTO):
    """C_i = A @ B_i^T for every weight B_i (all [N_i, K]) in one launch; returns
    the list of C_i."""
    torch = _torch()
    a_ptr, lda = _operand(A, "A")
    M, K = A.shape
    n = len(Bs)
    if Cs is None:
        Cs = []
        for B in Bs:
            ld = -(-B.shape[0] // 8) * 8
            Cs.append(torch.empty((M, ld), dtype=torch.bfloat16, device=A.device)[:, :B.shape[0]])
    if len(Cs) != n:
        raise ValueError("one output per weight")
    bp, nn, lb, cp, lc = ((ctypes.c_void_p * n)(), (ctypes.c_int64 * n)(), (ctypes.c_int64 * n)(),
                          (ctypes.c_void_p * n)(), (ctypes.c_int64 * n)())
    for i, (B, C) in enumerate(zip(Bs, Cs)):
        b_ptr, ldb = _operand(B, f"B[{i}]")
        c_ptr, ldc = _operand(C, f"C[{i}]")
        if B.shape[1] != K or tuple(C.shape) != (M, B.shape[0]):
            raise ValueError(f"shapes of B[{i}] {tuple(B.shape)} / C[{i}] {tuple(C.shape)}")
        bp[i], nn[i], lb[i], cp[i], lc[i] = b_ptr, B.shape[0], ldb, c_ptr, ldc
    with torch.cuda.device(A.device):
        st = load().gemv_bf16_batched(a_ptr, M, K, lda, bp, nn, lb, cp, lc, n, path, _stream_handle(stream))
    _check(st, "gemv_bf16_batched")
    return Cs


def gemv_bf16(A, B, C=None, stream=None, path: int = PATH_AUTO):
    """The skinny path (1 <= M <= 64); ``path`` picks the kernel (PATH_*)."""
    return _call("gemv_bf16", A, B, C, stream, path)


def gemv_bf16_noalloc(A, B, C=None, stream=None):
    """The CUDA-core skinny path with its scratch in the library's fixed device
    array instead of an allocated workspace (for callers that cannot allocate)."""
    return _call("gemv_bf16_noalloc", A, B, C, stream)


# ------------------------------------------------------------------ host-only helpers
def plan(M: int, N: int, K: int, num_sms: int, entry: int = 0) -> dict:
    info = PlanInfo()
    _check(load().sg_plan(M, N, K, num_sms, entry, ctypes.byref(info)), "sg_plan")
    d = info.as_dict()
    d["_struct"] = info
    return d


def plan_nvfp4(M: int, N: int, K: int, num_sms: int, path: int = PATH_AUTO) -> dict:
    info = PlanInfo()
    _check(load().sg_plan_nvfp4(M, N, K, num_sms, path, ctypes.byref(info)), "sg_plan_nvfp4")
    d = info.as_dict()
    d["_struct"] = info
    return d


def plan_swiglu(M: int, N: int, K: int, num_sms: int, entry: int = 0) -> dict:
    info = PlanInfo()
    _check(load().sg_plan_swiglu(M, N, K, num_sms, entry, ctypes.byref(info)), "sg_plan_swiglu")
    d = info.as_dict()
    d["_struct"] = info
    return d


def plan_items(info: dict) -> list[list[tuple]]:
    """All work items of a tcgen05 plan, per CTA: (tile, k0, k1, piece, npieces, slot, sk_index, tm, tn)."""
    lib = load()
    out = (ctypes.c_int32 * 9)()
    st = info["_struct"]
    items = []
    for cta in range(info["grid"]):
        row = []
        n = lib.sg_plan_item(ctypes.byref(st), cta, 0, out)
        for i in range(max(n, 0)):
            lib.sg_plan_item(ctypes.byref(st), cta, i, out)
            row.append(tuple(out))
        items.append(row)
    return items


def wave_efficiency(ctas: int, slots: int) -> float:
    return load().sg_wave_efficiency(ctas, slots)


def set_wait_timeout_ns(ns: int) -> None:
    load().sg_set_wait_timeout_ns(ns)


def check_device_errors(stream=None):
    """Synchronises the stream; returns (status, detail[4]) of kernel wait timeouts."""
    detail = (ctypes.c_uint32 * 4)()
    st = load().sg_check_device_errors(_stream_handle(stream), detail)
    return st, list(detail)


def device_query() -> dict:
    info = DeviceInfo()
    _check(load().sg_device_query(ctypes.byref(info)), "sg_device_query")
    return {name: getattr(info, name) for name, _ in info._fields_}


def bench_tcgen05_peak(iters: int, stream=None) -> tuple[float, float]:
    tf, mhz = ctypes.c_double(), ctypes.c_double()
    _check(load().sg_bench_tcgen05_peak(iters, ctypes.byref(tf), ctypes.byref(mhz), _stream_handle(stream)),
           "sg_bench_tcgen05_peak")
    return tf.value, mhz.value


def bench_copy(dst, src, reps: int = 20, stream=None) -> float:
    g = ctypes.c_double()
    nbytes = src.numel() * src.element_size()
    _check(load().sg_bench_copy(dst.data_ptr(), src.data_ptr(), nbytes, reps, ctypes.byref(g),
                                _stream_handle(stream)), "sg_bench_copy")
    return g.value


def bench_read(src, sink, reps: int = 20, stream=None) -> float:
    g = ctypes.c_double()
    nbytes = src.numel() * src.element_size()
    _check(load().sg_bench_read(src.data_ptr(), nbytes, reps, sink.data_ptr(), ctypes.byref(g),
                                _stream_handle(stream)), "sg_bench_read")
    return g.value
