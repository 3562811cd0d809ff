"""ctypes binding of ``libmoe.so`` (declared in ``include/moe.h``): argument marshalling only.

Every function takes torch CUDA tensors, passes their ``data_ptr()`` and the current CUDA
stream to the C entry point of the same name, and raises ``MoeError`` on a non-zero return.
All arithmetic happens in the library's kernels; there is no Python or CPU fallback — if the
library has not been built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_F = ctypes.c_float
_SIGS = {
    "moe_version": ([], _I),
    "moe_forward_launch_count": ([_I, _I, _I], _I),
    "moe_last_error_string": ([], ctypes.c_char_p),
    "moe_workspace_size": ([_I, _I, _I, _I, _I], _SZ),
    "moe_workspace_layout": ([_I, _I, _I, _I, _I, ctypes.POINTER(_SZ)], _I),
    "moe_host_staging_size": ([_I, _I, _I], _SZ),
    "moe_route": ([_P, _I, _I, _I, _P, _P, _P], _I),
    "moe_route_grouped": ([_P, _P, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, _P], _I),
    "moe_forward_grouped": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P, _SZ, _P],
                            _I),
    "moe_permute": ([_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_grouped_gemm_gateup_swiglu": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_grouped_gemm_gateup_swiglu_gather": ([_P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_grouped_gemm_down": ([_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_down_ksplit": ([_I, _I, _I, _I, _I], _I),
    "moe_gemm_pair_mode": ([_I, _I, _I, _I, _I, _I], _I),
    "moe_combine": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_forward_noalloc": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "moe_forward": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _SZ, _P], _I),
    "moe_forward_host": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _SZ, _P], _I),
    "moe_forward_host_batches": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P, _P, _P], _I),
    "moe_forward_fp8_host_batches": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P, _P, _P], _I),
    "moe_forward_fp8b_host_batches": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P, _P, _P], _I),
    "moe_forward_grouped_host_batches": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P, _SZ, _P,
                                          _P, _P], _I),
    "moe_forward_grouped_fp8_host_batches": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P,
                                              _SZ, _P, _P, _P], _I),
    "moe_forward_grouped_fp8b_host_batches": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _F, _P, _P,
                                               _SZ, _P, _P, _P], _I),
    "moe_get_device_error": ([_P, ctypes.POINTER(ctypes.c_int32)], _I),
    "moe_quantize_weights_fp8": ([_P, _I, _I, _I, _P, _P, _P], _I),
    "moe_permute_fp8": ([_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_quantize_rows_fp8": ([_P, _P, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_grouped_gemm_gateup_swiglu_fp8": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_grouped_gemm_down_fp8": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_workspace_size_fp8": ([_I, _I, _I, _I, _I], _SZ),
    "moe_workspace_layout_fp8": ([_I, _I, _I, _I, _I, ctypes.POINTER(_SZ)], _I),
    "moe_down_ksplit_fp8": ([_I, _I, _I, _I, _I], _I),
    "moe_gemm_pair_mode_fp8": ([_I, _I, _I, _I, _I, _I], _I),
    "moe_forward_fp8_launch_count": ([_I, _I, _I], _I),
    "moe_forward_fp8": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _SZ, _P], _I),
    "moe_quantize_weights_fp8b": ([_P, _I, _I, _I, _P, _P, _P], _I),
    "moe_quantize_rows_fp8b": ([_P, _P, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_grouped_gemm_gateup_swiglu_fp8b": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_grouped_gemm_gateup_swiglu_fp8b_q": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_fp8b_gemm_quantizes_h": ([_I, _I, _I], _I),
    "moe_grouped_gemm_down_fp8b": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_workspace_size_fp8b": ([_I, _I, _I, _I, _I], _SZ),
    "moe_workspace_layout_fp8b": ([_I, _I, _I, _I, _I, ctypes.POINTER(_SZ)], _I),
    "moe_down_ksplit_fp8b": ([_I, _I, _I, _I, _I], _I),
    "moe_forward_fp8b_launch_count": ([_I, _I, _I], _I),
    "moe_forward_fp8b": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _SZ, _P], _I),
    "moe_forward_grouped_fp8": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P,
                                 _SZ, _P], _I),
    "moe_forward_grouped_fp8b": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P, _P,
                                  _SZ, _P], _I),
}

WS_FIELDS = ("status", "idx", "w", "counts", "offsets", "src", "dest", "x_perm", "h", "y_perm", "total")
WS8_FIELDS = ("status", "idx", "w", "counts", "offsets", "src", "dest", "x8", "sx", "h", "h8", "sh", "y_perm",
              "total")

STATUS_BAD_EXPERT_ID = 0x1
STATUS_BAD_OFFSETS = 0x2
STATUS_BAD_DEST = 0x4
STATUS_WAIT_TIMEOUT = 0x8
STATUS_BAD_SRC = 0x10


class MoeError(RuntimeError):
    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} returned {code}: {msg}")
        self.code = code


_lock = threading.Lock()
_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load ``libmoe.so`` (once).  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with "
                                   "`python -m mixture_experts_grouped_fp32_gb300.build`")
            lib = ctypes.CDLL(path)
            for name, (args, res) in _SIGS.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _call(name: str, *args) -> None:
    L = load()
    rc = getattr(L, name)(*args)
    if rc != 0:
        raise MoeError(name, rc, L.moe_last_error_string().decode())


def _ptr(t: torch.Tensor | None):
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else stream


def _dev(t: torch.Tensor, dtype, name: str) -> None:
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor "
                         f"(got {t.dtype}, cuda={t.is_cuda}, contiguous={t.is_contiguous()})")


def workspace_size(T: int, d: int, f: int, E: int, top_k: int) -> int:
    return int(load().moe_workspace_size(T, d, f, E, top_k))


def workspace_layout(T: int, d: int, f: int, E: int, top_k: int) -> dict:
    out = (_SZ * 11)()
    _call("moe_workspace_layout", T, d, f, E, top_k, out)
    return dict(zip(WS_FIELDS, [int(v) for v in out]))


def host_staging_size(T: int, d: int, E: int) -> int:
    return int(load().moe_host_staging_size(T, d, E))


def forward_launch_count(T: int, E: int, top_k: int) -> int:
    """Kernel launches of one moe_forward call for this shape (4 with route+permute fused, else 5)."""
    return int(load().moe_forward_launch_count(T, E, top_k))


def route(logits: torch.Tensor, top_k: int, idx=None, w=None, stream=None):
    _dev(logits, torch.float32, "logits")
    T, E = logits.shape
    idx = idx if idx is not None else torch.empty(T, top_k, dtype=torch.int32, device=logits.device)
    w = w if w is not None else torch.empty(T, top_k, dtype=torch.float32, device=logits.device)
    _call("moe_route", _ptr(logits), T, E, top_k, _ptr(idx), _ptr(w), _stream(stream))
    return idx, w


def route_grouped(logits: torch.Tensor, bias: torch.Tensor, top_k: int, n_group: int, topk_group: int,
                  scale: float = 1.0, idx=None, w=None, stream=None):
    """DeepSeek-V3's router (sigmoid affinity, selection bias, group-limited top-k, scaled weights)."""
    _dev(logits, torch.float32, "logits")
    _dev(bias, torch.float32, "bias")
    T, E = logits.shape
    if bias.shape != (E,):
        raise ValueError(f"bias must have shape ({E},), got {tuple(bias.shape)}")
    idx = idx if idx is not None else torch.empty(T, top_k, dtype=torch.int32, device=logits.device)
    w = w if w is not None else torch.empty(T, top_k, dtype=torch.float32, device=logits.device)
    _call("moe_route_grouped", _ptr(logits), _ptr(bias), T, E, top_k, n_group, topk_group, float(scale), _ptr(idx),
          _ptr(w), _stream(stream))
    return idx, w


def permute(idx: torch.Tensor, x: torch.Tensor, E: int, status: torch.Tensor | None = None, stream=None,
            out: tuple | None = None):
    """Returns (counts, offsets, src, dest, x_perm); ``out`` may supply those five buffers."""
    _dev(idx, torch.int32, "idx")
    _dev(x, torch.bfloat16, "x")
    T, k = idx.shape
    d = x.shape[1]
    dev = x.device
    if out is not None:
        counts, offsets, src, dest, x_perm = out
    else:
        counts = torch.empty(E, dtype=torch.int32, device=dev)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        src = torch.empty(T * k, dtype=torch.int32, device=dev)
        dest = torch.empty(T, k, dtype=torch.int32, device=dev)
        x_perm = torch.empty(T * k, d, dtype=torch.bfloat16, device=dev)
    _call("moe_permute", _ptr(idx), _ptr(x), T, d, E, k, _ptr(counts), _ptr(offsets), _ptr(src),
          _ptr(dest), _ptr(x_perm), _ptr(status), _stream(stream))
    return counts, offsets, src, dest, x_perm


def grouped_gemm_gateup_swiglu(x_perm, w_gate_up, offsets, h=None, status=None, stream=None):
    _dev(x_perm, torch.bfloat16, "x_perm")
    _dev(w_gate_up, torch.bfloat16, "w_gate_up")
    _dev(offsets, torch.int32, "offsets")
    M, d = x_perm.shape
    E, _, f2 = w_gate_up.shape
    h = h if h is not None else torch.empty(M, f2 // 2, dtype=torch.bfloat16, device=x_perm.device)
    _call("moe_grouped_gemm_gateup_swiglu", _ptr(x_perm), _ptr(w_gate_up), _ptr(offsets), M, d, f2 // 2, E,
          _ptr(h), _ptr(status), _stream(stream))
    return h


def grouped_gemm_gateup_swiglu_gather(x, src, w_gate_up, offsets, h=None, status=None, stream=None):
    """Step 3 reading row r of the grouped operand as x[src[r]] (the kernel gathers the rows)."""
    _dev(x, torch.bfloat16, "x")
    _dev(src, torch.int32, "src")
    _dev(w_gate_up, torch.bfloat16, "w_gate_up")
    _dev(offsets, torch.int32, "offsets")
    T, d = x.shape
    M = src.numel()
    E, _, f2 = w_gate_up.shape
    h = h if h is not None else torch.empty(M, f2 // 2, dtype=torch.bfloat16, device=x.device)
    _call("moe_grouped_gemm_gateup_swiglu_gather", _ptr(x), _ptr(src), T, _ptr(w_gate_up), _ptr(offsets), M, d,
          f2 // 2, E, _ptr(h), _ptr(status), _stream(stream))
    return h


def down_ksplit(T: int, d: int, f: int, E: int, top_k: int) -> int:
    """K slices moe_forward uses for the down projection of this shape."""
    return int(load().moe_down_ksplit(T, d, f, E, top_k))


def gemm_pair_mode(T: int, d: int, f: int, E: int, top_k: int, kind: int = 0) -> int:
    """Grouped-GEMM kernel moe_forward picks for this shape and GEMM (kind 0 gate+up, 1 down):
    0 single SMs, 1 SM pairs with 256-row tiles only, 2 SM pairs that also swap small experts;
    -1 for an invalid shape."""
    return int(load().moe_gemm_pair_mode(T, d, f, E, top_k, kind))


def grouped_gemm_down(h, w_down, offsets, y_perm=None, status=None, stream=None, ksplit: int = 1):
    """y_perm [ksplit, M, d] fp32 partial sums (a [M, d] view when ksplit == 1)."""
    _dev(h, torch.bfloat16, "h")
    _dev(w_down, torch.bfloat16, "w_down")
    _dev(offsets, torch.int32, "offsets")
    M, f = h.shape
    E, _, d = w_down.shape
    if y_perm is None:
        y_perm = torch.empty(ksplit, M, d, dtype=torch.float32, device=h.device)
        if ksplit == 1:
            y_perm = y_perm[0]
    if y_perm.numel() < ksplit * M * d:
        raise ValueError("y_perm must hold ksplit * M * d floats")
    _call("moe_grouped_gemm_down", _ptr(h), _ptr(w_down), _ptr(offsets), M, d, f, E, ksplit, _ptr(y_perm),
          _ptr(status), _stream(stream))
    return y_perm


def combine(y_perm, w, dest, out=None, status=None, stream=None, ksplit: int = 1):
    """y_perm is [T*k, d] or [ksplit, T*k, d] partial sums; out bf16 [T, d]."""
    _dev(y_perm, torch.float32, "y_perm")
    _dev(w, torch.float32, "w")
    _dev(dest, torch.int32, "dest")
    T, k = dest.shape
    d = y_perm.shape[-1]
    if y_perm.numel() < ksplit * T * k * d:
        raise ValueError("y_perm must hold ksplit * T * k * d floats")
    out = out if out is not None else torch.empty(T, d, dtype=torch.bfloat16, device=y_perm.device)
    _call("moe_combine", _ptr(y_perm), _ptr(w), _ptr(dest), T, d, k, ksplit, _ptr(out), _ptr(status),
          _stream(stream))
    return out


def forward(x, logits, w_gate_up, w_down, top_k, out=None, workspace=None, stream=None):
    """One call for the whole layer (five kernel launches).  Returns ``out`` bf16 [T, d]."""
    _dev(x, torch.bfloat16, "x")
    _dev(logits, torch.float32, "logits")
    _dev(w_gate_up, torch.bfloat16, "w_gate_up")
    _dev(w_down, torch.bfloat16, "w_down")
    T, d = x.shape
    E, _, f2 = w_gate_up.shape
    if workspace is None:
        workspace = torch.empty(workspace_size(T, d, f2 // 2, E, top_k), dtype=torch.uint8, device=x.device)
    out = out if out is not None else torch.empty(T, d, dtype=torch.bfloat16, device=x.device)
    _call("moe_forward", _ptr(x), _ptr(logits), _ptr(w_gate_up), _ptr(w_down), T, d, f2 // 2, E, top_k,
          _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    return out


def forward_grouped(x, logits, bias, w_gate_up, w_down, top_k, n_group, topk_group, scale=1.0, out=None,
                    workspace=None, stream=None):
    """The layer with DeepSeek-V3's router as step 1 (five kernel launches).  Returns ``out``."""
    _dev(x, torch.bfloat16, "x")
    _dev(logits, torch.float32, "logits")
    _dev(bias, torch.float32, "bias")
    _dev(w_gate_up, torch.bfloat16, "w_gate_up")
    _dev(w_down, torch.bfloat16, "w_down")
    T, d = x.shape
    E, _, f2 = w_gate_up.shape
    if workspace is None:
        workspace = torch.empty(workspace_size(T, d, f2 // 2, E, top_k), dtype=torch.uint8, device=x.device)
    out = out if out is not None else torch.empty(T, d, dtype=torch.bfloat16, device=x.device)
    _call("moe_forward_grouped", _ptr(x), _ptr(logits), _ptr(bias), _ptr(w_gate_up), _ptr(w_down), T, d, f2 // 2,
          E, top_k, n_group, topk_group, float(scale), _ptr(out), _ptr(workspace), workspace.numel(),
          _stream(stream))
    return out


def forward_host(x_host, logits_host, w_gate_up, w_down, top_k, out_host, workspace, stream=None):
    """The layer with x, logits and out in (page-locked) host memory; copies are enqueued on the
    stream together with the five kernels.  Synchronise the stream before reading ``out_host``."""
    for t, n in ((x_host, "x_host"), (logits_host, "logits_host"), (out_host, "out_host")):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous host tensor")
    _dev(w_gate_up, torch.bfloat16, "w_gate_up")
    _dev(w_down, torch.bfloat16, "w_down")
    T, d = x_host.shape
    E, _, f2 = w_gate_up.shape
    _call("moe_forward_host", _ptr(x_host), _ptr(logits_host), _ptr(w_gate_up), _ptr(w_down), T, d, f2 // 2, E,
          top_k, _ptr(out_host), _ptr(workspace), workspace.numel(), _stream(stream))
    return out_host


def forward_host_batches(x_hosts, logits_hosts, w_gate_up, w_down, top_k, out_hosts, workspace, stream=None,
                         h2d_stream=None, d2h_stream=None):
    """The layer over a list of batches in (page-locked) host memory, copies overlapped with the
    layers: the layers run on ``stream``, the copies on ``h2d_stream`` / ``d2h_stream`` (created
    here when not given).  The workspace holds workspace_size() + 2 * host_staging_size() bytes.
    Synchronise ``stream`` before reading ``out_hosts``."""
    if len(x_hosts) == 0:
        return out_hosts
    _dev(w_gate_up, torch.bfloat16, "w_gate_up")
    _dev(w_down, torch.bfloat16, "w_down")
    E, _, f2 = w_gate_up.shape
    n, T, d, xa, la, oa, h2d, d2h = _host_batch_args(x_hosts, logits_hosts, out_hosts, w_gate_up.device,
                                                     h2d_stream, d2h_stream)
    _call("moe_forward_host_batches", xa, la, _ptr(w_gate_up), _ptr(w_down), n, T, d, f2 // 2, E, top_k, oa,
          _ptr(workspace), workspace.numel(), _stream(stream), _stream(h2d), _stream(d2h))
    return out_hosts


def _host_batch_args(x_hosts, logits_hosts, out_hosts, device, h2d_stream, d2h_stream):
    n = len(x_hosts)
    if len(logits_hosts) != n or len(out_hosts) != n:
        raise ValueError("x_hosts, logits_hosts and out_hosts must have one tensor per batch")
    T, d = x_hosts[0].shape
    for i in range(n):
        for t, nm, shape in ((x_hosts[i], "x_hosts", (T, d)), (logits_hosts[i], "logits_hosts", None),
                             (out_hosts[i], "out_hosts", (T, d))):
            if t.is_cuda or not t.is_contiguous() or (shape is not None and tuple(t.shape) != shape):
                raise ValueError(f"{nm}[{i}] must be a contiguous host tensor of the first batch's shape")
    h2d = h2d_stream if h2d_stream is not None else torch.cuda.Stream(device=device)
    d2h = d2h_stream if d2h_stream is not None else torch.cuda.Stream(device=device)
    arr = lambda ts: (ctypes.c_void_p * n)(*[t.data_ptr() for t in ts])
    return n, T, d, arr(x_hosts), arr(logits_hosts), arr(out_hosts), h2d, d2h


def _forward8_host_batches(sym, x_hosts, logits_hosts, w8_gate_up, s_gate_up, w8_down, s_down, top_k, out_hosts,
                           workspace, stream, h2d_stream, d2h_stream):
    if len(x_hosts) == 0:
        return out_hosts
    E, f2, _ = _w8_dims(w8_gate_up, "w8_gate_up")
    n, T, d, xa, la, oa, h2d, d2h = _host_batch_args(x_hosts, logits_hosts, out_hosts, w8_gate_up.device,
                                                     h2d_stream, d2h_stream)
    _call(sym, xa, la, _ptr(w8_gate_up), _ptr(s_gate_up), _ptr(w8_down), _ptr(s_down), n, T, d, f2 // 2, E, top_k,
          oa, _ptr(workspace), workspace.numel(), _stream(stream), _stream(h2d), _stream(d2h))
    return out_hosts


def forward_fp8_host_batches(x_hosts, logits_hosts, w8_gate_up, s_gate_up, w8_down, s_down, top_k, out_hosts,
                             workspace, stream=None, h2d_stream=None, d2h_stream=None):
    """forward_host_batches with the FP8 layer (per-row / per-channel scales); the workspace holds
    workspace_size_fp8() + 2 * host_staging_size() bytes."""
    return _forward8_host_batches("moe_forward_fp8_host_batches", x_hosts, logits_hosts, w8_gate_up, s_gate_up,
                                  w8_down, s_down, top_k, out_hosts, workspace, stream, h2d_stream, d2h_stream)


def forward_fp8b_host_batches(x_hosts, logits_hosts, w8_gate_up, s_gate_up, w8_down, s_down, top_k, out_hosts,
                              workspace, stream=None, h2d_stream=None, d2h_stream=None):
    """forward_host_batches with the blockwise FP8 layer; the workspace holds workspace_size_fp8b() +
    2 * host_staging_size() bytes."""
    return _forward8_host_batches("moe_forward_fp8b_host_batches", x_hosts, logits_hosts, w8_gate_up, s_gate_up,
                                  w8_down, s_down, top_k, out_hosts, workspace, stream, h2d_stream, d2h_stream)


def forward_grouped_host_batches(x_hosts, logits_hosts, bias, w_gate_up, w_down, top_k, n_group, topk_group, scale,
                                 out_hosts, workspace, stream=None, h2d_stream=None, d2h_stream=None):
    """forward_host_batches with DeepSeek-V3's router (bias [E] fp32 on the device)."""
    if len(x_hosts) == 0:
        return out_hosts
    _dev(w_gate_up, torch.bfloat16, "w_gate_up")
    _dev(w_down, torch.bfloat16, "w_down")
    _dev(bias, torch.float32, "bias")
    E, _, f2 = w_gate_up.shape
    n, T, d, xa, la, oa, h2d, d2h = _host_batch_args(x_hosts, logits_hosts, out_hosts, w_gate_up.device,
                                                     h2d_stream, d2h_stream)
    _call("moe_forward_grouped_host_batches", xa, la, _ptr(bias), _ptr(w_gate_up), _ptr(w_down), n, T, d, f2 // 2, E,
          top_k, n_group, topk_group, float(scale), oa, _ptr(workspace), workspace.numel(), _stream(stream),
          _stream(h2d), _stream(d2h))
    return out_hosts


def forward_grouped_fp8_host_batches(x_hosts, logits_hosts, bias, w8_gate_up, s_gate_up, w8_down, s_down, top_k,
                                     n_group, topk_group, scale, out_hosts, workspace, stream=None, h2d_stream=None,
                                     d2h_stream=None, blocks: bool = False):
    """The FP8 layers (blocks=True: block scales) over host batches with DeepSeek-V3's router."""
    if len(x_hosts) == 0:
        return out_hosts
    _dev(bias, torch.float32, "bias")
    E, f2, _ = _w8_dims(w8_gate_up, "w8_gate_up")
    n, T, d, xa, la, oa, h2d, d2h = _host_batch_args(x_hosts, logits_hosts, out_hosts, w8_gate_up.device,
                                                     h2d_stream, d2h_stream)
    sym = "moe_forward_grouped_fp8b_host_batches" if blocks else "moe_forward_grouped_fp8_host_batches"
    _call(sym, xa, la, _ptr(bias), _ptr(w8_gate_up), _ptr(s_gate_up), _ptr(w8_down), _ptr(s_down), n, T, d, f2 // 2,
          E, top_k, n_group, topk_group, float(scale), oa, _ptr(workspace), workspace.numel(), _stream(stream),
          _stream(h2d), _stream(d2h))
    return out_hosts


def get_device_error(status_or_workspace: torch.Tensor) -> int:
    code = ctypes.c_int32(0)
    _call("moe_get_device_error", _ptr(status_or_workspace), ctypes.byref(code))
    return int(code.value)


def workspace_views(ws: torch.Tensor, T: int, d: int, f: int, E: int, top_k: int) -> dict:
    """Typed views of moe_forward's intermediates inside ``ws`` (for inspection and tests)."""
    L = workspace_layout(T, d, f, E, top_k)
    M = T * top_k
    S = down_ksplit(T, d, f, E, top_k)

    def view(name, n, dtype, shape):
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return ws[L[name]:L[name] + nbytes].view(dtype).view(*shape)

    return {
        "status": view("status", 1, torch.int32, (1,)),
        "idx": view("idx", M, torch.int32, (T, top_k)),
        "w": view("w", M, torch.float32, (T, top_k)),
        "counts": view("counts", E, torch.int32, (E,)),
        "offsets": view("offsets", E + 1, torch.int32, (E + 1,)),
        "src": view("src", M, torch.int32, (M,)),
        "dest": view("dest", M, torch.int32, (T, top_k)),
        "x_perm": view("x_perm", M * d, torch.bfloat16, (M, d)),
        "h": view("h", M * f, torch.bfloat16, (M, f)),
        "y_perm": view("y_perm", S * M * d, torch.float32, (S, M, d)),
        "ksplit": S,
    }


class MoELayer:
    """A Mixture-of-Experts FFN layer whose weights and workspace live on one GPU.

    ``layer(x, logits)`` runs the five-kernel forward on the current stream and returns bf16
    [T, d]; the workspace grows on demand and is reused across calls."""

    def __init__(self, w_gate_up: torch.Tensor, w_down: torch.Tensor, top_k: int):
        _dev(w_gate_up, torch.bfloat16, "w_gate_up")
        _dev(w_down, torch.bfloat16, "w_down")
        self.w_gate_up, self.w_down, self.top_k = w_gate_up, w_down, top_k
        self.E, self.d, f2 = w_gate_up.shape
        self.f = f2 // 2
        self._ws = torch.empty(0, dtype=torch.uint8, device=w_gate_up.device)

    def workspace(self, T: int) -> torch.Tensor:
        need = workspace_size(T, self.d, self.f, self.E, self.top_k)
        if self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=self.w_gate_up.device)
        return self._ws

    def __call__(self, x: torch.Tensor, logits: torch.Tensor, out: torch.Tensor | None = None):
        return forward(x, logits, self.w_gate_up, self.w_down, self.top_k, out=out,
                       workspace=self.workspace(x.shape[0]))


# ---------------------------------------------------------------------------------------------
# FP8 (E4M3) variant: codes are torch.uint8 tensors, scales float32.
# ---------------------------------------------------------------------------------------------
def quantize_weights_fp8(W: torch.Tensor, stream=None, out: tuple | None = None):
    """W [E, K, N] bf16 -> (Wq uint8 E4M3 codes [E, N/64, K/128, 64, 128], scale [E, N] fp32): the
    transposed codes in 8 KB blocks of 64 output columns x 128 K (see ``fp8_unblock``), one scale
    per output column (absmax over K / 448)."""
    _dev(W, torch.bfloat16, "W")
    E, K, N = W.shape
    Wq, scale = out if out is not None else (
        torch.empty(E, N // 64, K // 128, 64, 128, dtype=torch.uint8, device=W.device),
        torch.empty(E, N, dtype=torch.float32, device=W.device))
    _call("moe_quantize_weights_fp8", _ptr(W), E, K, N, _ptr(Wq), _ptr(scale), _stream(stream))
    return Wq, scale


def _w8_dims(w8: torch.Tensor, name: str):
    """(E, N, K) of blocked FP8 weight codes [E, N/64, K/128, 64, 128]."""
    _dev(w8, torch.uint8, name)
    if w8.dim() != 5 or w8.shape[3:] != (64, 128):
        raise ValueError(f"{name} must be blocked FP8 codes [E, N/64, K/128, 64, 128], got {tuple(w8.shape)}")
    return w8.shape[0], w8.shape[1] * 64, w8.shape[2] * 128


def fp8_unblock(w8):
    """Blocked codes [E, N/64, K/128, 64, 128] (tensor or array) -> [E, N, K] (index work only)."""
    E, G, B = w8.shape[:3]
    return w8.transpose(2, 3).reshape(E, G * 64, B * 128) if isinstance(w8, torch.Tensor) else \
        w8.transpose(0, 1, 3, 2, 4).reshape(E, G * 64, B * 128)


def fp8_block(w):
    """[E, N, K] codes (tensor or array) -> the blocked layout [E, N/64, K/128, 64, 128]."""
    E, N, K = w.shape
    v = w.reshape(E, N // 64, 64, K // 128, 128)
    return v.transpose(2, 3).contiguous() if isinstance(w, torch.Tensor) else \
        v.transpose(0, 1, 3, 2, 4).copy()


def permute_fp8(idx: torch.Tensor, x: torch.Tensor, E: int, status: torch.Tensor | None = None, stream=None,
                out: tuple | None = None):
    """Step 2 of the FP8 layer: returns (counts, offsets, src, dest, x8_perm, sx) with x8_perm [T*k, d]
    uint8 E4M3 codes and sx [T*k] fp32; ``out`` may supply those six buffers."""
    _dev(idx, torch.int32, "idx")
    _dev(x, torch.bfloat16, "x")
    T, k = idx.shape
    d = x.shape[1]
    dev = x.device
    if out is not None:
        counts, offsets, src, dest, x8, sx = out
    else:
        counts = torch.empty(E, dtype=torch.int32, device=dev)
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
        src = torch.empty(T * k, dtype=torch.int32, device=dev)
        dest = torch.empty(T, k, dtype=torch.int32, device=dev)
        x8 = torch.empty(T * k, d, dtype=torch.uint8, device=dev)
        sx = torch.empty(T * k, dtype=torch.float32, device=dev)
    _call("moe_permute_fp8", _ptr(idx), _ptr(x), T, d, E, k, _ptr(counts), _ptr(offsets), _ptr(src), _ptr(dest),
          _ptr(x8), _ptr(sx), _ptr(status), _stream(stream))
    return counts, offsets, src, dest, x8, sx


def quantize_rows_fp8(a: torch.Tensor, src: torch.Tensor | None = None, status=None, stream=None,
                      out: tuple | None = None):
    """Rows of a [R0, C] bf16 (row src[r] for output row r when src is given) -> (codes [R, C] uint8,
    scale [R] fp32)."""
    _dev(a, torch.bfloat16, "a")
    if src is not None:
        _dev(src, torch.int32, "src")
    R0, C = a.shape
    R = R0 if src is None else src.numel()
    q, scale = out if out is not None else (torch.empty(R, C, dtype=torch.uint8, device=a.device),
                                            torch.empty(R, dtype=torch.float32, device=a.device))
    _call("moe_quantize_rows_fp8", _ptr(a), _ptr(src), R, C, R0, _ptr(q), _ptr(scale), _ptr(status),
          _stream(stream))
    return q, scale


def grouped_gemm_gateup_swiglu_fp8(x8_perm, sx, w8_gate_up, s_gate_up, offsets, h=None, status=None, stream=None):
    """Step 3 on E4M3 codes: x8_perm [M, d] uint8 + sx [M]; w8_gate_up [E, 2f, d] uint8 + s_gate_up [E, 2f]."""
    _dev(x8_perm, torch.uint8, "x8_perm")
    _dev(sx, torch.float32, "sx")
    _dev(s_gate_up, torch.float32, "s_gate_up")
    _dev(offsets, torch.int32, "offsets")
    M, d = x8_perm.shape
    E, f2, _ = _w8_dims(w8_gate_up, "w8_gate_up")
    h = h if h is not None else torch.empty(M, f2 // 2, dtype=torch.bfloat16, device=x8_perm.device)
    _call("moe_grouped_gemm_gateup_swiglu_fp8", _ptr(x8_perm), _ptr(sx), _ptr(w8_gate_up), _ptr(s_gate_up),
          _ptr(offsets), M, d, f2 // 2, E, _ptr(h), _ptr(status), _stream(stream))
    return h


def grouped_gemm_down_fp8(h8, sh, w8_down, s_down, offsets, y_perm=None, status=None, stream=None, ksplit: int = 1):
    """Step 4 on E4M3 codes: h8 [M, f] uint8 + sh [M]; w8_down [E, d, f] uint8 + s_down [E, d]."""
    _dev(h8, torch.uint8, "h8")
    _dev(sh, torch.float32, "sh")
    _dev(s_down, torch.float32, "s_down")
    _dev(offsets, torch.int32, "offsets")
    M, f = h8.shape
    E, d, _ = _w8_dims(w8_down, "w8_down")
    if y_perm is None:
        y_perm = torch.empty(ksplit, M, d, dtype=torch.float32, device=h8.device)
        if ksplit == 1:
            y_perm = y_perm[0]
    if y_perm.numel() < ksplit * M * d:
        raise ValueError("y_perm must hold ksplit * M * d floats")
    _call("moe_grouped_gemm_down_fp8", _ptr(h8), _ptr(sh), _ptr(w8_down), _ptr(s_down), _ptr(offsets), M, d, f, E,
          ksplit, _ptr(y_perm), _ptr(status), _stream(stream))
    return y_perm


def workspace_size_fp8(T: int, d: int, f: int, E: int, top_k: int) -> int:
    return int(load().moe_workspace_size_fp8(T, d, f, E, top_k))


def workspace_layout_fp8(T: int, d: int, f: int, E: int, top_k: int) -> dict:
    out = (_SZ * 14)()
    _call("moe_workspace_layout_fp8", T, d, f, E, top_k, out)
    return dict(zip(WS8_FIELDS, [int(v) for v in out]))


def down_ksplit_fp8(T: int, d: int, f: int, E: int, top_k: int) -> int:
    return int(load().moe_down_ksplit_fp8(T, d, f, E, top_k))


def gemm_pair_mode_fp8(T: int, d: int, f: int, E: int, top_k: int, kind: int = 0) -> int:
    """As gemm_pair_mode, for moe_forward_fp8's grouped GEMMs."""
    return int(load().moe_gemm_pair_mode_fp8(T, d, f, E, top_k, kind))


def forward_fp8_launch_count(T: int, E: int, top_k: int) -> int:
    """Kernel launches of one moe_forward_fp8 call (5 with route+permute fused, else 6)."""
    return int(load().moe_forward_fp8_launch_count(T, E, top_k))


def forward_fp8(x, logits, w8_gate_up, s_gate_up, w8_down, s_down, top_k, out=None, workspace=None, stream=None):
    """The FP8 layer in one call.  Weights as returned by quantize_weights_fp8 of w_gate_up [E, d, 2f]
    and w_down [E, f, d].  Returns ``out`` bf16 [T, d]."""
    _dev(x, torch.bfloat16, "x")
    _dev(logits, torch.float32, "logits")
    _dev(s_gate_up, torch.float32, "s_gate_up")
    _dev(s_down, torch.float32, "s_down")
    T, d = x.shape
    E, f2, _ = _w8_dims(w8_gate_up, "w8_gate_up")
    _w8_dims(w8_down, "w8_down")
    if workspace is None:
        workspace = torch.empty(workspace_size_fp8(T, d, f2 // 2, E, top_k), dtype=torch.uint8, device=x.device)
    out = out if out is not None else torch.empty(T, d, dtype=torch.bfloat16, device=x.device)
    _call("moe_forward_fp8", _ptr(x), _ptr(logits), _ptr(w8_gate_up), _ptr(s_gate_up), _ptr(w8_down), _ptr(s_down),
          T, d, f2 // 2, E, top_k, _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    return out


def workspace_views_fp8(ws: torch.Tensor, T: int, d: int, f: int, E: int, top_k: int) -> dict:
    """Typed views of moe_forward_fp8's intermediates inside ``ws``."""
    L = workspace_layout_fp8(T, d, f, E, top_k)
    M = T * top_k
    S = down_ksplit_fp8(T, d, f, E, top_k)

    def view(name, n, dtype, shape):
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return ws[L[name]:L[name] + nbytes].view(dtype).view(*shape)

    return {
        "status": view("status", 1, torch.int32, (1,)),
        "idx": view("idx", M, torch.int32, (T, top_k)),
        "w": view("w", M, torch.float32, (T, top_k)),
        "counts": view("counts", E, torch.int32, (E,)),
        "offsets": view("offsets", E + 1, torch.int32, (E + 1,)),
        "src": view("src", M, torch.int32, (M,)),
        "dest": view("dest", M, torch.int32, (T, top_k)),
        "x8": view("x8", M * d, torch.uint8, (M, d)),
        "sx": view("sx", M, torch.float32, (M,)),
        "h": view("h", M * f, torch.bfloat16, (M, f)),
        "h8": view("h8", M * f, torch.uint8, (M, f)),
        "sh": view("sh", M, torch.float32, (M,)),
        "y_perm": view("y_perm", S * M * d, torch.float32, (S, M, d)),
        "ksplit": S,
    }


# ---------------------------------------------------------------------------------------------
# Blockwise FP8: 1 x 128 activation blocks, 128 x 128 weight blocks, power-of-two scales.
# ---------------------------------------------------------------------------------------------
def quantize_weights_fp8b(W: torch.Tensor, stream=None, out: tuple | None = None):
    """W [E, K, N] bf16 -> (Wq blocked codes [E, N/64, K/128, 64, 128], scale [E, N/128, K/128])."""
    _dev(W, torch.bfloat16, "W")
    E, K, N = W.shape
    Wq, scale = out if out is not None else (
        torch.empty(E, N // 64, K // 128, 64, 128, dtype=torch.uint8, device=W.device),
        torch.empty(E, N // 128, K // 128, dtype=torch.float32, device=W.device))
    _call("moe_quantize_weights_fp8b", _ptr(W), E, K, N, _ptr(Wq), _ptr(scale), _stream(stream))
    return Wq, scale


def quantize_rows_fp8b(a: torch.Tensor, src: torch.Tensor | None = None, status=None, stream=None,
                       out: tuple | None = None):
    """Rows of a [R0, C] bf16 in 128-wide blocks -> (codes [R, C] uint8, scale [R, C/128] fp32)."""
    _dev(a, torch.bfloat16, "a")
    if src is not None:
        _dev(src, torch.int32, "src")
    R0, C = a.shape
    R = R0 if src is None else src.numel()
    q, scale = out if out is not None else (torch.empty(R, C, dtype=torch.uint8, device=a.device),
                                            torch.empty(R, C // 128, dtype=torch.float32, device=a.device))
    _call("moe_quantize_rows_fp8b", _ptr(a), _ptr(src), R, C, R0, _ptr(q), _ptr(scale), _ptr(status),
          _stream(stream))
    return q, scale


def grouped_gemm_gateup_swiglu_fp8b(x8_perm, sx, w8_gate_up, s_gate_up, offsets, h=None, status=None, stream=None):
    """Blockwise step 3: sx [M, d/128], s_gate_up [E, 2f/128, d/128]."""
    _dev(x8_perm, torch.uint8, "x8_perm")
    _dev(sx, torch.float32, "sx")
    _dev(s_gate_up, torch.float32, "s_gate_up")
    _dev(offsets, torch.int32, "offsets")
    M, d = x8_perm.shape
    E, f2, _ = _w8_dims(w8_gate_up, "w8_gate_up")
    h = h if h is not None else torch.empty(M, f2 // 2, dtype=torch.bfloat16, device=x8_perm.device)
    _call("moe_grouped_gemm_gateup_swiglu_fp8b", _ptr(x8_perm), _ptr(sx), _ptr(w8_gate_up), _ptr(s_gate_up),
          _ptr(offsets), M, d, f2 // 2, E, _ptr(h), _ptr(status), _stream(stream))
    return h


def grouped_gemm_gateup_swiglu_fp8b_q(x8_perm, sx, w8_gate_up, s_gate_up, offsets, h8=None, sh=None, status=None,
                                      stream=None):
    """Blockwise step 3 with h quantised in the epilogue: (h8 [M, f] codes, sh [M, f/128] scales)."""
    _dev(x8_perm, torch.uint8, "x8_perm")
    _dev(sx, torch.float32, "sx")
    _dev(s_gate_up, torch.float32, "s_gate_up")
    _dev(offsets, torch.int32, "offsets")
    M, d = x8_perm.shape
    E, f2, _ = _w8_dims(w8_gate_up, "w8_gate_up")
    f = f2 // 2
    h8 = h8 if h8 is not None else torch.empty(M, f, dtype=torch.uint8, device=x8_perm.device)
    sh = sh if sh is not None else torch.empty(M, f // 128, dtype=torch.float32, device=x8_perm.device)
    _call("moe_grouped_gemm_gateup_swiglu_fp8b_q", _ptr(x8_perm), _ptr(sx), _ptr(w8_gate_up), _ptr(s_gate_up),
          _ptr(offsets), M, d, f, E, _ptr(h8), _ptr(sh), _ptr(status), _stream(stream))
    return h8, sh


def grouped_gemm_down_fp8b(h8, sh, w8_down, s_down, offsets, y_perm=None, status=None, stream=None, ksplit: int = 1):
    """Blockwise step 4: sh [M, f/128], s_down [E, d/128, f/128]."""
    _dev(h8, torch.uint8, "h8")
    _dev(sh, torch.float32, "sh")
    _dev(s_down, torch.float32, "s_down")
    _dev(offsets, torch.int32, "offsets")
    M, f = h8.shape
    E, d, _ = _w8_dims(w8_down, "w8_down")
    if y_perm is None:
        y_perm = torch.empty(ksplit, M, d, dtype=torch.float32, device=h8.device)
        if ksplit == 1:
            y_perm = y_perm[0]
    if y_perm.numel() < ksplit * M * d:
        raise ValueError("y_perm must hold ksplit * M * d floats")
    _call("moe_grouped_gemm_down_fp8b", _ptr(h8), _ptr(sh), _ptr(w8_down), _ptr(s_down), _ptr(offsets), M, d, f, E,
          ksplit, _ptr(y_perm), _ptr(status), _stream(stream))
    return y_perm


def workspace_size_fp8b(T: int, d: int, f: int, E: int, top_k: int) -> int:
    return int(load().moe_workspace_size_fp8b(T, d, f, E, top_k))


def workspace_layout_fp8b(T: int, d: int, f: int, E: int, top_k: int) -> dict:
    out = (_SZ * 14)()
    _call("moe_workspace_layout_fp8b", T, d, f, E, top_k, out)
    return dict(zip(WS8_FIELDS, [int(v) for v in out]))


def down_ksplit_fp8b(T: int, d: int, f: int, E: int, top_k: int) -> int:
    return int(load().moe_down_ksplit_fp8b(T, d, f, E, top_k))


def forward_fp8b_launch_count(T: int, E: int, top_k: int) -> int:
    """Kernel launches of one moe_forward_fp8b call (5 or 6 with route+permute fused, one more
    otherwise; see fp8b_gemm_quantizes_h)."""
    return int(load().moe_forward_fp8b_launch_count(T, E, top_k))


def fp8b_gemm_quantizes_h(T: int, E: int, top_k: int) -> bool:
    """Whether moe_forward_fp8b's gate+up GEMM quantises h itself (T*top_k > 64*E, or MOE_FP8B_FUSE_H)."""
    return int(load().moe_fp8b_gemm_quantizes_h(T, E, top_k)) == 1


def forward_fp8b(x, logits, w8_gate_up, s_gate_up, w8_down, s_down, top_k, out=None, workspace=None, stream=None):
    """The blockwise FP8 layer in one call (weights from quantize_weights_fp8b).  Returns ``out``."""
    _dev(x, torch.bfloat16, "x")
    _dev(logits, torch.float32, "logits")
    _dev(s_gate_up, torch.float32, "s_gate_up")
    _dev(s_down, torch.float32, "s_down")
    T, d = x.shape
    E, f2, _ = _w8_dims(w8_gate_up, "w8_gate_up")
    _w8_dims(w8_down, "w8_down")
    if workspace is None:
        workspace = torch.empty(workspace_size_fp8b(T, d, f2 // 2, E, top_k), dtype=torch.uint8, device=x.device)
    out = out if out is not None else torch.empty(T, d, dtype=torch.bfloat16, device=x.device)
    _call("moe_forward_fp8b", _ptr(x), _ptr(logits), _ptr(w8_gate_up), _ptr(s_gate_up), _ptr(w8_down), _ptr(s_down),
          T, d, f2 // 2, E, top_k, _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    return out


def workspace_views_fp8b(ws: torch.Tensor, T: int, d: int, f: int, E: int, top_k: int) -> dict:
    """Typed views of moe_forward_fp8b's intermediates inside ``ws``."""
    L = workspace_layout_fp8b(T, d, f, E, top_k)
    M = T * top_k
    S = down_ksplit_fp8b(T, d, f, E, top_k)

    def view(name, n, dtype, shape):
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return ws[L[name]:L[name] + nbytes].view(dtype).view(*shape)

    return {
        "status": view("status", 1, torch.int32, (1,)),
        "idx": view("idx", M, torch.int32, (T, top_k)),
        "w": view("w", M, torch.float32, (T, top_k)),
        "counts": view("counts", E, torch.int32, (E,)),
        "offsets": view("offsets", E + 1, torch.int32, (E + 1,)),
        "src": view("src", M, torch.int32, (M,)),
        "dest": view("dest", M, torch.int32, (T, top_k)),
        "x8": view("x8", M * d, torch.uint8, (M, d)),
        "sx": view("sx", M * (d // 128), torch.float32, (M, d // 128)),
        "h": view("h", M * f, torch.bfloat16, (M, f)),
        "h8": view("h8", M * f, torch.uint8, (M, f)),
        "sh": view("sh", M * (f // 128), torch.float32, (M, f // 128)),
        "y_perm": view("y_perm", S * M * d, torch.float32, (S, M, d)),
        "ksplit": S,
    }


def forward_grouped_fp8(x, logits, bias, w8_gate_up, s_gate_up, w8_down, s_down, top_k, n_group, topk_group,
                        scale=1.0, out=None, workspace=None, stream=None, blocks: bool = False):
    """An FP8 layer (per-row / per-channel scales, or blockwise with ``blocks``) with DeepSeek-V3's
    router as step 1.  Weights as returned by quantize_weights_fp8 / quantize_weights_fp8b."""
    _dev(x, torch.bfloat16, "x")
    _dev(logits, torch.float32, "logits")
    _dev(bias, torch.float32, "bias")
    _dev(s_gate_up, torch.float32, "s_gate_up")
    _dev(s_down, torch.float32, "s_down")
    T, d = x.shape
    E, f2, _ = _w8_dims(w8_gate_up, "w8_gate_up")
    _w8_dims(w8_down, "w8_down")
    if workspace is None:
        size = workspace_size_fp8b if blocks else workspace_size_fp8
        workspace = torch.empty(size(T, d, f2 // 2, E, top_k), dtype=torch.uint8, device=x.device)
    out = out if out is not None else torch.empty(T, d, dtype=torch.bfloat16, device=x.device)
    _call("moe_forward_grouped_fp8b" if blocks else "moe_forward_grouped_fp8", _ptr(x), _ptr(logits), _ptr(bias),
          _ptr(w8_gate_up), _ptr(s_gate_up), _ptr(w8_down), _ptr(s_down), T, d, f2 // 2, E, top_k, n_group,
          topk_group, float(scale), _ptr(out), _ptr(workspace), workspace.numel(), _stream(stream))
    return out
