"""CPU oracle for the Mixture-of-Experts FFN layer forward — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference legs may
import this package.  The product library (``libmoe.so`` and its Python binding) never imports
it, and the two share no code: this wrapper loads ``liboracle.so`` built from
``moe_oracle.cpp`` with the host C++ compiler.

Arrays are numpy, C-contiguous; bf16 tensors travel as ``uint16`` bit patterns.
The arithmetic, its sources and its readings of the pages are documented in ``moe_oracle.cpp``.
Every function here is pinned by ``tests/test_oracle_pins.py`` (closed forms, a hand-worked
example, library routines, a float64 brute force and the layer's invariants).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: no fused multiply-add contraction, so x86 and Arm builds round alike.
CXXFLAGS = ["-O3", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared"]


def build(src: str = _SRC, out: str = _LIB, extra: list[str] | None = None) -> str:
    """Compile the oracle shared library (``g++``).  Returns the path of the built library."""
    cmd = ["g++", *CXXFLAGS, *(extra or []), src, "-o", out + ".tmp"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    os.replace(out + ".tmp", out)
    return out


def _needs_build() -> bool:
    return not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)


_I32P = ctypes.POINTER(ctypes.c_int32)
_F32P = ctypes.POINTER(ctypes.c_float)
_U16P = ctypes.POINTER(ctypes.c_uint16)
_U8P = ctypes.POINTER(ctypes.c_uint8)
_INT = ctypes.c_int

_SIGS = {
    "oracle_num_threads": ([], _INT),
    "oracle_route": ([_F32P, _INT, _INT, _INT, _I32P, _F32P], _INT),
    "oracle_permute": ([_I32P, _INT, _INT, _INT, _I32P, _I32P, _I32P, _I32P], _INT),
    "oracle_gather_rows": ([_U16P, _I32P, _INT, _INT, _U16P], None),
    "oracle_gateup_swiglu": ([_U16P, _I32P, _INT, _U16P, _INT, _INT, _F32P], None),
    "oracle_down": ([_F32P, _I32P, _INT, _U16P, _INT, _INT, _F32P], None),
    "oracle_down_bf16": ([_U16P, _I32P, _INT, _U16P, _INT, _INT, _F32P], None),
    "oracle_combine": ([_F32P, _F32P, _I32P, _INT, _INT, _INT, _F32P], None),
    "oracle_forward": ([_U16P, _F32P, _U16P, _U16P, _INT, _INT, _INT, _INT, _INT, _F32P], _INT),
    "oracle_forward_tokens": ([_U16P, _F32P, _U16P, _U16P, _INT, _INT, _INT, _INT, _INT, _I32P, _INT,
                               _F32P], _INT),
    "oracle_route_grouped": ([_F32P, _F32P, _INT, _INT, _INT, _INT, _INT, ctypes.c_float, _I32P, _F32P], _INT),
    "oracle_forward_routed": ([_U16P, _I32P, _F32P, _U16P, _U16P, _INT, _INT, _INT, _INT, _INT, _F32P], _INT),
    "oracle_forward_tokens_routed": ([_U16P, _I32P, _F32P, _U16P, _U16P, _INT, _INT, _INT, _INT, _INT, _I32P,
                                      _INT, _F32P], _INT),
    "oracle_e4m3_encode_array": ([_F32P, _INT, _U8P], None),
    "oracle_e4m3_decode_array": ([_U8P, _INT, _F32P], None),
    "oracle_quantize_rows_fp8": ([_U16P, _INT, _INT, _U8P, _F32P], None),
    "oracle_quantize_weights_fp8": ([_U16P, _INT, _INT, _INT, _U8P, _F32P], None),
    "oracle_gateup_swiglu_fp8": ([_U8P, _F32P, _I32P, _INT, _U8P, _F32P, _INT, _INT, _U16P], None),
    "oracle_pow2_block_scale": ([ctypes.c_float], ctypes.c_float),
    "oracle_quantize_rows_fp8b": ([_U16P, _INT, _INT, _U8P, _F32P], None),
    "oracle_quantize_weights_fp8b": ([_U16P, _INT, _INT, _INT, _U8P, _F32P], None),
    "oracle_forward_fp8b_tokens_routed": ([_U16P, _I32P, _F32P, _U8P, _F32P, _U8P, _F32P, _INT, _INT, _INT, _INT,
                                           _INT, _I32P, _INT, _F32P], _INT),
    "oracle_gateup_swiglu_fp8b": ([_U8P, _F32P, _I32P, _INT, _U8P, _F32P, _INT, _INT, _U16P], None),
    "oracle_down_fp8b": ([_U8P, _F32P, _I32P, _INT, _U8P, _F32P, _INT, _INT, _F32P], None),
    "oracle_down_fp8": ([_U8P, _F32P, _I32P, _INT, _U8P, _F32P, _INT, _INT, _F32P], None),
    "oracle_forward_fp8_tokens_routed": ([_U16P, _I32P, _F32P, _U8P, _F32P, _U8P, _F32P, _INT, _INT, _INT, _INT,
                                          _INT, _I32P, _INT, _F32P], _INT),
}


def load_library(path: str) -> ctypes.CDLL:
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            if _needs_build():
                build()
            _lib = load_library(_LIB)
    return _lib


def _p(a: np.ndarray, ptype):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ptype)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


class Oracle:
    """Thin numpy wrapper over one loaded oracle library (the default one, or a test's build)."""

    def __init__(self, library: ctypes.CDLL | None = None):
        self.L = library if library is not None else lib()

    def num_threads(self) -> int:
        return int(self.L.oracle_num_threads())

    def route(self, logits, k):
        logits = _c(logits, np.float32)
        T, E = logits.shape
        idx = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float32)
        rc = self.L.oracle_route(_p(logits, _F32P), T, E, k, _p(idx, _I32P), _p(w, _F32P))
        if rc:
            raise ValueError(f"oracle_route rejected the shape (rc={rc})")
        return idx, w

    def permute(self, idx, E):
        idx = _c(idx, np.int32)
        T, k = idx.shape
        counts = np.empty(E, np.int32)
        offsets = np.empty(E + 1, np.int32)
        src = np.empty(T * k, np.int32)
        dest = np.empty((T, k), np.int32)
        rc = self.L.oracle_permute(_p(idx, _I32P), T, E, k, _p(counts, _I32P), _p(offsets, _I32P),
                                   _p(src, _I32P), _p(dest, _I32P))
        if rc:
            raise ValueError(f"oracle_permute rejected its input (rc={rc})")
        return counts, offsets, src, dest

    def gather_rows(self, x_bits, src):
        x_bits = _c(x_bits, np.uint16)
        src = _c(src, np.int32)
        M, d = src.shape[0], x_bits.shape[1]
        out = np.empty((M, d), np.uint16)
        self.L.oracle_gather_rows(_p(x_bits, _U16P), _p(src, _I32P), M, d, _p(out, _U16P))
        return out

    def gateup_swiglu(self, x_perm_bits, offsets, wgu_bits):
        x_perm_bits = _c(x_perm_bits, np.uint16)
        offsets = _c(offsets, np.int32)
        wgu_bits = _c(wgu_bits, np.uint16)
        E, d, f2 = wgu_bits.shape
        f = f2 // 2
        M = x_perm_bits.shape[0]
        h = np.zeros((M, f), np.float32)
        self.L.oracle_gateup_swiglu(_p(x_perm_bits, _U16P), _p(offsets, _I32P), E,
                                    _p(wgu_bits, _U16P), d, f, _p(h, _F32P))
        return h

    def down(self, h, offsets, wd_bits):
        offsets = _c(offsets, np.int32)
        wd_bits = _c(wd_bits, np.uint16)
        E, f, d = wd_bits.shape
        M = h.shape[0]
        y = np.zeros((M, d), np.float32)
        if h.dtype == np.uint16:
            h = _c(h, np.uint16)
            self.L.oracle_down_bf16(_p(h, _U16P), _p(offsets, _I32P), E, _p(wd_bits, _U16P), d, f,
                                    _p(y, _F32P))
        else:
            h = _c(h, np.float32)
            self.L.oracle_down(_p(h, _F32P), _p(offsets, _I32P), E, _p(wd_bits, _U16P), d, f,
                               _p(y, _F32P))
        return y

    def combine(self, y, w, dest):
        y = _c(y, np.float32)
        w = _c(w, np.float32)
        dest = _c(dest, np.int32)
        T, k = dest.shape
        d = y.shape[1]
        out = np.empty((T, d), np.float32)
        self.L.oracle_combine(_p(y, _F32P), _p(w, _F32P), _p(dest, _I32P), T, d, k, _p(out, _F32P))
        return out

    def forward(self, x_bits, logits, wgu_bits, wd_bits, k):
        x_bits = _c(x_bits, np.uint16)
        logits = _c(logits, np.float32)
        wgu_bits = _c(wgu_bits, np.uint16)
        wd_bits = _c(wd_bits, np.uint16)
        T, d = x_bits.shape
        E, _, f2 = wgu_bits.shape
        out = np.empty((T, d), np.float32)
        rc = self.L.oracle_forward(_p(x_bits, _U16P), _p(logits, _F32P), _p(wgu_bits, _U16P),
                                   _p(wd_bits, _U16P), T, d, f2 // 2, E, k, _p(out, _F32P))
        if rc:
            raise ValueError(f"oracle_forward failed (rc={rc})")
        return out

    def forward_tokens(self, x_bits, logits, wgu_bits, wd_bits, k, tokens):
        x_bits = _c(x_bits, np.uint16)
        logits = _c(logits, np.float32)
        wgu_bits = _c(wgu_bits, np.uint16)
        wd_bits = _c(wd_bits, np.uint16)
        tokens = _c(tokens, np.int32)
        T, d = x_bits.shape
        E, _, f2 = wgu_bits.shape
        out = np.empty((tokens.shape[0], d), np.float32)
        rc = self.L.oracle_forward_tokens(_p(x_bits, _U16P), _p(logits, _F32P), _p(wgu_bits, _U16P),
                                          _p(wd_bits, _U16P), T, d, f2 // 2, E, k,
                                          _p(tokens, _I32P), tokens.shape[0], _p(out, _F32P))
        if rc:
            raise ValueError(f"oracle_forward_tokens failed (rc={rc})")
        return out

    def route_grouped(self, logits, bias, k, n_group, topk_group, scale=1.0):
        """DeepSeek-V3 router: sigmoid affinities, selection bias, group-limited top-k."""
        logits = _c(logits, np.float32)
        bias = _c(bias, np.float32)
        T, E = logits.shape
        assert bias.shape == (E,)
        idx = np.empty((T, k), np.int32)
        w = np.empty((T, k), np.float32)
        rc = self.L.oracle_route_grouped(_p(logits, _F32P), _p(bias, _F32P), T, E, k, n_group, topk_group,
                                         float(scale), _p(idx, _I32P), _p(w, _F32P))
        if rc:
            raise ValueError(f"oracle_route_grouped rejected the shape (rc={rc})")
        return idx, w

    def forward_routed(self, x_bits, idx, w, wgu_bits, wd_bits):
        """Steps 2-5 of the layer for a given routing idx/w [T,k]."""
        x_bits = _c(x_bits, np.uint16)
        idx = _c(idx, np.int32)
        w = _c(w, np.float32)
        wgu_bits = _c(wgu_bits, np.uint16)
        wd_bits = _c(wd_bits, np.uint16)
        T, d = x_bits.shape
        E, _, f2 = wgu_bits.shape
        k = idx.shape[1]
        out = np.empty((T, d), np.float32)
        rc = self.L.oracle_forward_routed(_p(x_bits, _U16P), _p(idx, _I32P), _p(w, _F32P), _p(wgu_bits, _U16P),
                                          _p(wd_bits, _U16P), T, d, f2 // 2, E, k, _p(out, _F32P))
        if rc:
            raise ValueError(f"oracle_forward_routed failed (rc={rc})")
        return out

    def forward_tokens_routed(self, x_bits, idx_rows, w_rows, wgu_bits, wd_bits, tokens):
        """The layer's output for the sampled tokens, given their routing idx_rows/w_rows [ntok,k]."""
        x_bits = _c(x_bits, np.uint16)
        idx_rows = _c(idx_rows, np.int32)
        w_rows = _c(w_rows, np.float32)
        wgu_bits = _c(wgu_bits, np.uint16)
        wd_bits = _c(wd_bits, np.uint16)
        tokens = _c(tokens, np.int32)
        T, d = x_bits.shape
        E, _, f2 = wgu_bits.shape
        k = idx_rows.shape[1]
        out = np.empty((tokens.shape[0], d), np.float32)
        rc = self.L.oracle_forward_tokens_routed(_p(x_bits, _U16P), _p(idx_rows, _I32P), _p(w_rows, _F32P),
                                                 _p(wgu_bits, _U16P), _p(wd_bits, _U16P), T, d, f2 // 2, E, k,
                                                 _p(tokens, _I32P), tokens.shape[0], _p(out, _F32P))
        if rc:
            raise ValueError(f"oracle_forward_tokens_routed failed (rc={rc})")
        return out

    # ---- FP8 variant ----
    def e4m3_encode(self, x):
        x = _c(x, np.float32)
        out = np.empty(x.shape, np.uint8)
        self.L.oracle_e4m3_encode_array(_p(x.reshape(-1), _F32P), x.size, _p(out.reshape(-1), _U8P))
        return out

    def e4m3_decode(self, codes):
        codes = _c(codes, np.uint8)
        out = np.empty(codes.shape, np.float32)
        self.L.oracle_e4m3_decode_array(_p(codes.reshape(-1), _U8P), codes.size, _p(out.reshape(-1), _F32P))
        return out

    def quantize_rows_fp8(self, a_bits):
        a_bits = _c(a_bits, np.uint16)
        R, C = a_bits.shape
        q = np.empty((R, C), np.uint8)
        sc = np.empty(R, np.float32)
        self.L.oracle_quantize_rows_fp8(_p(a_bits, _U16P), R, C, _p(q, _U8P), _p(sc, _F32P))
        return q, sc

    def quantize_weights_fp8(self, w_bits):
        """W [E, K, N] bf16 bits -> (codes [E, N, K], scales [E, N])."""
        w_bits = _c(w_bits, np.uint16)
        E, K, N = w_bits.shape
        q = np.empty((E, N, K), np.uint8)
        sc = np.empty((E, N), np.float32)
        self.L.oracle_quantize_weights_fp8(_p(w_bits, _U16P), E, K, N, _p(q, _U8P), _p(sc, _F32P))
        return q, sc

    def gateup_swiglu_fp8(self, x8_perm, sx, offsets, wgu8, sgu):
        """FP8 step 3: codes x8_perm [M, d] + sx [M], wgu8 [E, 2f, d] + sgu [E, 2f] -> h [M, f] bf16 bits
        (rows past offsets[E] zero)."""
        x8_perm, sx = _c(x8_perm, np.uint8), _c(sx, np.float32)
        offsets = _c(offsets, np.int32)
        wgu8, sgu = _c(wgu8, np.uint8), _c(sgu, np.float32)
        E, f2, d = wgu8.shape
        M = x8_perm.shape[0]
        h = np.zeros((M, f2 // 2), np.uint16)
        self.L.oracle_gateup_swiglu_fp8(_p(x8_perm, _U8P), _p(sx, _F32P), _p(offsets, _I32P), E, _p(wgu8, _U8P),
                                        _p(sgu, _F32P), d, f2 // 2, _p(h, _U16P))
        return h

    def down_fp8(self, h8, sh, offsets, wd8, sd):
        """FP8 step 4: codes h8 [M, f] + sh [M], wd8 [E, d, f] + sd [E, d] -> y [M, d] fp32."""
        h8, sh = _c(h8, np.uint8), _c(sh, np.float32)
        offsets = _c(offsets, np.int32)
        wd8, sd = _c(wd8, np.uint8), _c(sd, np.float32)
        E, d, f = wd8.shape
        M = h8.shape[0]
        y = np.zeros((M, d), np.float32)
        self.L.oracle_down_fp8(_p(h8, _U8P), _p(sh, _F32P), _p(offsets, _I32P), E, _p(wd8, _U8P), _p(sd, _F32P), d,
                               f, _p(y, _F32P))
        return y

    def forward_fp8_tokens_routed(self, x_bits, idx_rows, w_rows, wgu8, sgu, wd8, sd, tokens):
        x_bits = _c(x_bits, np.uint16)
        idx_rows = _c(idx_rows, np.int32)
        w_rows = _c(w_rows, np.float32)
        wgu8, wd8 = _c(wgu8, np.uint8), _c(wd8, np.uint8)
        sgu, sd = _c(sgu, np.float32), _c(sd, np.float32)
        tokens = _c(tokens, np.int32)
        T, d = x_bits.shape
        E, f2, _ = wgu8.shape
        k = idx_rows.shape[1]
        out = np.empty((tokens.shape[0], d), np.float32)
        rc = self.L.oracle_forward_fp8_tokens_routed(
            _p(x_bits, _U16P), _p(idx_rows, _I32P), _p(w_rows, _F32P), _p(wgu8, _U8P), _p(sgu, _F32P),
            _p(wd8, _U8P), _p(sd, _F32P), T, d, f2 // 2, E, k, _p(tokens, _I32P), tokens.shape[0], _p(out, _F32P))
        if rc:
            raise ValueError(f"oracle_forward_fp8_tokens_routed failed (rc={rc})")
        return out

    def forward_fp8(self, x_bits, logits, wgu8, sgu, wd8, sd, k):
        """The whole FP8 layer with the softmax router (every token)."""
        idx, w = self.route(logits, k)
        T = idx.shape[0]
        return self.forward_fp8_tokens_routed(x_bits, idx, w, wgu8, sgu, wd8, sd, np.arange(T, dtype=np.int32))


    # ---- blockwise FP8 (1 x 128 activation blocks, 128 x 128 weight blocks, power-of-two scales) ----
    def pow2_block_scale(self, amax: float) -> float:
        return float(self.L.oracle_pow2_block_scale(float(amax)))

    def quantize_rows_fp8b(self, a_bits):
        """[R, C] bf16 bits -> (codes [R, C], block scales [R, C/128])."""
        a_bits = _c(a_bits, np.uint16)
        R, C = a_bits.shape
        q = np.empty((R, C), np.uint8)
        sc = np.empty((R, C // 128), np.float32)
        self.L.oracle_quantize_rows_fp8b(_p(a_bits, _U16P), R, C, _p(q, _U8P), _p(sc, _F32P))
        return q, sc

    def quantize_weights_fp8b(self, w_bits):
        """W [E, K, N] bf16 bits -> (codes [E, N, K], block scales [E, N/128, K/128])."""
        w_bits = _c(w_bits, np.uint16)
        E, K, N = w_bits.shape
        q = np.empty((E, N, K), np.uint8)
        sc = np.empty((E, N // 128, K // 128), np.float32)
        self.L.oracle_quantize_weights_fp8b(_p(w_bits, _U16P), E, K, N, _p(q, _U8P), _p(sc, _F32P))
        return q, sc

    def gateup_swiglu_fp8b(self, x8_perm, sx, offsets, wgu8, sgu):
        x8_perm, sx = _c(x8_perm, np.uint8), _c(sx, np.float32)
        offsets = _c(offsets, np.int32)
        wgu8, sgu = _c(wgu8, np.uint8), _c(sgu, np.float32)
        E, f2, d = wgu8.shape
        M = x8_perm.shape[0]
        h = np.zeros((M, f2 // 2), np.uint16)
        self.L.oracle_gateup_swiglu_fp8b(_p(x8_perm, _U8P), _p(sx, _F32P), _p(offsets, _I32P), E, _p(wgu8, _U8P),
                                         _p(sgu, _F32P), d, f2 // 2, _p(h, _U16P))
        return h

    def down_fp8b(self, h8, sh, offsets, wd8, sd):
        h8, sh = _c(h8, np.uint8), _c(sh, np.float32)
        offsets = _c(offsets, np.int32)
        wd8, sd = _c(wd8, np.uint8), _c(sd, np.float32)
        E, d, f = wd8.shape
        M = h8.shape[0]
        y = np.zeros((M, d), np.float32)
        self.L.oracle_down_fp8b(_p(h8, _U8P), _p(sh, _F32P), _p(offsets, _I32P), E, _p(wd8, _U8P), _p(sd, _F32P), d,
                                f, _p(y, _F32P))
        return y

    def forward_fp8b_tokens_routed(self, x_bits, idx_rows, w_rows, wgu8, sgu, wd8, sd, tokens):
        x_bits = _c(x_bits, np.uint16)
        idx_rows = _c(idx_rows, np.int32)
        w_rows = _c(w_rows, np.float32)
        wgu8, wd8 = _c(wgu8, np.uint8), _c(wd8, np.uint8)
        sgu, sd = _c(sgu, np.float32), _c(sd, np.float32)
        tokens = _c(tokens, np.int32)
        T, d = x_bits.shape
        E, f2, _ = wgu8.shape
        k = idx_rows.shape[1]
        out = np.empty((tokens.shape[0], d), np.float32)
        rc = self.L.oracle_forward_fp8b_tokens_routed(
            _p(x_bits, _U16P), _p(idx_rows, _I32P), _p(w_rows, _F32P), _p(wgu8, _U8P), _p(sgu, _F32P),
            _p(wd8, _U8P), _p(sd, _F32P), T, d, f2 // 2, E, k, _p(tokens, _I32P), tokens.shape[0], _p(out, _F32P))
        if rc:
            raise ValueError(f"oracle_forward_fp8b_tokens_routed failed (rc={rc})")
        return out

    def forward_fp8b(self, x_bits, logits, wgu8, sgu, wd8, sd, k):
        """The whole blockwise FP8 layer with the softmax router (every token)."""
        idx, w = self.route(logits, k)
        T = idx.shape[0]
        return self.forward_fp8b_tokens_routed(x_bits, idx, w, wgu8, sgu, wd8, sd, np.arange(T, dtype=np.int32))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)
