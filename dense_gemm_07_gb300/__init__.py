"""dense_gemm_07_gb300 -- dense GEMM C = A*B on one NVIDIA GB300 (sm_103a).

The computation lives in hand-written CUDA kernels behind the C ABI of
``libgemm07.so`` (declared in ``include/gemm07.h``).  This package is the thin
Python binding: the names below match the C entry points and only marshal
torch tensors into (sizes, pointers, leading dimensions, stream).  PyTorch
provides device memory and streams; it computes nothing on this path, and a
missing or unloadable library is an error, never a fallback.

    import dense_gemm_07_gb300 as g7
    C = g7.gemm_bf16_f32acc(A_bf16, B_bf16)   # A: MxK, B: KxN, CUDA tensors
    C = g7.gemm_f32(A_f32, B_f32)

The raw ctypes entry points (integer addresses) are in ``dense_gemm_07_gb300.abi``.
"""
from __future__ import annotations

from . import _abi as abi
from ._build import build

__all__ = ["abi", "build", "GemmError", "gemm_f32", "gemm_bf16_f32acc", "gemm_f32_ladder",
           "gemm_f32_ex", "gemm_bf16_f32acc_ex",
           "gemm_f32_host", "gemm_bf16_f32acc_host", "gemm_get_device_status",
           "gemm_status_string", "plan"]


class GemmError(RuntimeError):
    """A nonzero gemm_status_t from the library."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {abi.gemm_status_string(status)} (status {status})")


def gemm_status_string(status: int) -> str:
    return abi.gemm_status_string(status)


def _torch():
    import torch
    return torch


def _ld(t, rows_name: str) -> int:
    """Row stride of a 2-D tensor whose rows are contiguous and do not
    overlap (a broadcast row, stride 0, would be read past its storage)."""
    rows, cols = t.shape
    if cols > 1 and t.stride(1) != 1:
        raise ValueError(f"{rows_name}: rows must be contiguous (stride(1) == 1)")
    if rows > 1 and cols > 0 and t.stride(0) < cols:
        raise ValueError(f"{rows_name}: rows must not overlap (stride(0) >= columns)")
    return max(t.stride(0) if rows > 1 else cols, cols, 1)


def _ptr(t) -> int | None:
    return t.data_ptr() if t.numel() else None


def _operands(A, B, dtype, out, device_kind: str):
    torch = _torch()
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("A and B must be 2-D")
    if A.dtype != dtype or B.dtype != dtype:
        raise TypeError(f"A and B must be {dtype}")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner sizes differ: A is {M}x{K}, B is {K2}x{N}")
    dev = A.device
    if device_kind == "cuda":
        if dev.type != "cuda" or B.device != dev:
            raise ValueError("A and B must be CUDA tensors on the same device")
    elif dev.type != "cpu" or B.device.type != "cpu":
        raise ValueError("host variant: A and B must be CPU tensors")
    if out is None:
        pin = device_kind == "cpu" and torch.cuda.is_available()
        out = torch.empty((M, N), dtype=torch.float32, device=dev, pin_memory=pin) \
            if device_kind == "cpu" else torch.empty((M, N), dtype=torch.float32, device=dev)
    else:
        if out.shape != (M, N) or out.dtype != torch.float32 or out.device != dev:
            raise ValueError("out must be an M x N float32 tensor on A's device")
    return M, N, K, out


def _stream_handle(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _call(fn_name, dtype, A, B, out, stream, device_kind):
    torch = _torch()
    M, N, K, out = _operands(A, B, dtype, out, device_kind)
    dev = A.device if device_kind == "cuda" else torch.device("cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        s = getattr(abi, fn_name)(M, N, K, _ptr(A), _ld(A, "A"), _ptr(B), _ld(B, "B"),
                                  _ptr(out), _ld(out, "out"), _stream_handle(stream, dev))
    if s != abi.GEMM_OK:
        raise GemmError(s, fn_name)
    return out


def gemm_f32(A, B, out=None, stream=None):
    """C = A @ B for float32 CUDA tensors on the FP32 CUDA-core kernel."""
    return _call("gemm_f32", _torch().float32, A, B, out, stream, "cuda")


def gemm_bf16_f32acc(A, B, out=None, stream=None):
    """C = A @ B for bfloat16 CUDA tensors; FP32 accumulation and output."""
    return _call("gemm_bf16_f32acc", _torch().bfloat16, A, B, out, stream, "cuda")


def _gemm_ex(fn_name, dtype, A, B, out, alpha, beta, bias, activation, stream):
    torch = _torch()
    if beta != 0.0 and out is None:
        raise ValueError("beta != 0 reads C: pass its prior contents as `out`")
    M, N, K, out = _operands(A, B, dtype, out, "cuda")
    acts = {"none": abi.ACT_NONE, "relu": abi.ACT_RELU, "gelu": abi.ACT_GELU}
    if activation not in acts:
        raise ValueError(f"activation must be one of {sorted(acts)}")
    if bias is not None:
        if bias.shape != (N,) or bias.dtype != torch.float32 or bias.device != A.device \
                or (N > 1 and bias.stride(0) != 1):
            raise ValueError("bias must be a contiguous float32 vector of N elements "
                             "on A's device")
    epi = abi.GemmEpilogue(float(alpha), float(beta),
                           bias.data_ptr() if bias is not None and bias.numel() else None,
                           acts[activation])
    with torch.cuda.device(A.device):
        s = getattr(abi, fn_name)(M, N, K, _ptr(A), _ld(A, "A"), _ptr(B), _ld(B, "B"),
                                  _ptr(out), _ld(out, "out"), epi,
                                  _stream_handle(stream, A.device))
    if s != abi.GEMM_OK:
        raise GemmError(s, fn_name)
    return out


def gemm_f32_ex(A, B, out=None, alpha=1.0, beta=0.0, bias=None, activation="none",
                stream=None):
    """C = act(alpha * A @ B + beta * C + bias) for float32 CUDA tensors."""
    return _gemm_ex("gemm_f32_ex", _torch().float32, A, B, out, alpha, beta, bias,
                    activation, stream)


def gemm_bf16_f32acc_ex(A, B, out=None, alpha=1.0, beta=0.0, bias=None,
                        activation="none", stream=None):
    """C = act(alpha * A @ B + beta * C + bias) for bfloat16 A, B; FP32 C."""
    return _gemm_ex("gemm_bf16_f32acc_ex", _torch().bfloat16, A, B, out, alpha, beta,
                    bias, activation, stream)


def gemm_f32_ladder(rung, A, B, out=None, stream=None):
    """C = A @ B with teaching rung 0, 1 or 2 (FP32, for measurement)."""
    torch = _torch()
    M, N, K, out = _operands(A, B, torch.float32, out, "cuda")
    with torch.cuda.device(A.device):
        s = abi.gemm_f32_ladder(int(rung), M, N, K, _ptr(A), _ld(A, "A"), _ptr(B),
                                _ld(B, "B"), _ptr(out), _ld(out, "out"),
                                _stream_handle(stream, A.device))
    if s != abi.GEMM_OK:
        raise GemmError(s, "gemm_f32_ladder")
    return out


def gemm_f32_host(A, B, out=None, stream=None):
    """Host-buffer variant of gemm_f32: CPU tensors in and out (synchronous)."""
    return _call("gemm_f32_host", _torch().float32, A, B, out, stream, "cpu")


def gemm_bf16_f32acc_host(A, B, out=None, stream=None):
    """Host-buffer variant of gemm_bf16_f32acc (synchronous)."""
    return _call("gemm_bf16_f32acc_host", _torch().bfloat16, A, B, out, stream, "cpu")


def gemm_get_device_status(stream=None) -> int:
    """Sync the stream and read/clear the device status word (0 = OK)."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device())
    return abi.gemm_get_device_status(_stream_handle(stream, dev))


def plan(kind: str, M, N, K, A=16, lda=None, B=16, ldb=None, C=16, ldc=None):
    """Path the entry point takes for these sizes/addresses (no GPU needed)."""
    lda = max(K, 1) if lda is None else lda
    ldb = max(N, 1) if ldb is None else ldb
    ldc = max(N, 1) if ldc is None else ldc
    fn = abi.gemm_plan_bf16 if kind == "bf16" else abi.gemm_plan_f32
    s, p = fn(M, N, K, A, lda, B, ldb, C, ldc)
    return s, p
