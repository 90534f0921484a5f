"""Thin ctypes binding of libgdn.so (include/gdn.h).

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels.  Torch tensors are accepted for convenience and passed as raw
device pointers; the current torch stream is used unless one is given.  If
the library is missing the import fails loudly: there is no other path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

GDN_OK = 0
GDN_F32 = 0
GDN_BF16 = 1
FLAG_SEQLENS = 0x1
FLAG_BLOCK_RANGE = 0x2
FLAG_TRASH_WRITE = 0x4
FLAG_DUPLICATE = 0x8
FLAG_TIMEOUT = 0x10
FLAG_HINT = 0x20
FLAG_RANGE = 0x40

EXPORTED = [
    "gdn_state_pool_layout_for",
    "gdn_state_pool_create",
    "gdn_state_pool_destroy",
    "gdn_state_pool_layout",
    "gdn_state_pool_copy_block",
    "gdn_state_pool_reserve",
    "gdn_varlen_forward",
    "gdn_varlen_forward_noalloc",
    "gdn_kda_varlen_forward",
    "gdn_ssd_pool_layout_for",
    "gdn_ssd_pool_create",
    "gdn_ssd_varlen_forward",
    "gdn_get_error",
    "gdn_pool_set_timing_events",
    "gdn_prefill_scratch_bytes", "gdn_pool_last_prefill_path",
    "gdn_in_proj",
    "gdn_out_proj",
    "gdn_status_string",
]

PREFILL_NONE, PREFILL_SPLIT, PREFILL_FUSED, PREFILL_SERIAL = 0, 1, 2, 3


class GdnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class Weights(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("A_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p)]


class SsdWeights(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("A_log", ctypes.c_void_p),
                ("dt_bias", ctypes.c_void_p), ("D", ctypes.c_void_p)]


_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def load() -> ctypes.CDLL:
    """Load libgdn.so (it must have been built by build())."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise ImportError(f"libgdn.so not built at {path}: run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    PS = ctypes.POINTER(ctypes.c_size_t)
    lib.gdn_state_pool_layout_for.argtypes = [I] * 8 + [S, PS, PS, PS, PS]
    lib.gdn_state_pool_create.argtypes = [ctypes.POINTER(P)] + [I] * 8 + [S, P, S]
    lib.gdn_state_pool_destroy.argtypes = [P]
    lib.gdn_state_pool_layout.argtypes = [P, PS, PS, PS, ctypes.POINTER(P)]
    lib.gdn_state_pool_copy_block.argtypes = [P, I, I, I, P]
    lib.gdn_state_pool_reserve.argtypes = [P, I]
    lib.gdn_varlen_forward.argtypes = [P, I, P, P, P, P, P, P, ctypes.POINTER(Weights), P,
                                       I, I, I, P]
    lib.gdn_kda_varlen_forward.argtypes = lib.gdn_varlen_forward.argtypes
    lib.gdn_ssd_pool_layout_for.argtypes = [I] * 8 + [S, PS, PS, PS, PS]
    lib.gdn_ssd_pool_create.argtypes = [ctypes.POINTER(P)] + [I] * 8 + [S, P, S]
    lib.gdn_ssd_varlen_forward.argtypes = [P, I, P, P, P, P, P, ctypes.POINTER(SsdWeights), P,
                                           I, I, I, P]
    lib.gdn_varlen_forward_noalloc.argtypes = [P, S] + [I] * 8 + [S, I] + [P] * 6 + [
        ctypes.POINTER(Weights), P, I, I, I, P, P]
    lib.gdn_get_error.argtypes = [P, I, ctypes.POINTER(ctypes.c_uint32), I, P]
    lib.gdn_pool_set_timing_events.argtypes = [P, P, P]
    lib.gdn_pool_last_prefill_path.argtypes = [P, ctypes.POINTER(ctypes.c_int)]
    lib.gdn_prefill_scratch_bytes.argtypes = [I] * 6 + [PS]
    lib.gdn_in_proj.argtypes = [P, I, I, P, P, P, P, I, I, I, P, P, P, P, P, P]
    lib.gdn_out_proj.argtypes = [P, P, P, ctypes.c_float, P, I, I, I, I, P, P, P, P]
    lib.gdn_diag_umma_gemm.argtypes = [P, P, P, P, I, I, I, P]
    lib.gdn_diag_umma_gemm.restype = I
    lib.gdn_diag_umma_gemm_ex.argtypes = [P, P, P, P, I, I, I, I, I, P]
    lib.gdn_diag_umma_gemm_ex.restype = I
    lib.gdn_diag_wait_timeout.argtypes = [P, P]
    lib.gdn_diag_wait_timeout.restype = I
    lib.gdn_status_string.argtypes = [I]
    lib.gdn_status_string.restype = ctypes.c_char_p
    for name in EXPORTED[:-1]:
        getattr(lib, name).restype = I
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().gdn_status_string(status).decode()


def _check(status: int, what: str):
    if status != GDN_OK:
        raise GdnError(status, what)


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def act_code(dtype) -> int:
    if dtype in (torch.float32, "f32"):
        return GDN_F32
    if dtype in (torch.bfloat16, "bf16"):
        return GDN_BF16
    raise ValueError(f"unsupported activation dtype {dtype}")


def layout_for(num_blocks, num_layers, Hk, Hv, dk, dv, K, act, block_align=0):
    """(block_stride, conv_off, rec_off, total_bytes) without allocating."""
    out = [ctypes.c_size_t() for _ in range(4)]
    _check(load().gdn_state_pool_layout_for(num_blocks, num_layers, Hk, Hv, dk, dv, K,
                                            act_code(act), block_align,
                                            *[ctypes.byref(o) for o in out]),
           "gdn_state_pool_layout_for")
    return tuple(o.value for o in out)


def ssd_layout_for(num_blocks, num_layers, H, P, N, G, K, act, block_align=0):
    """(block_stride, conv_off, ssm_off, total_bytes) of a Mamba2 pool."""
    out = [ctypes.c_size_t() for _ in range(4)]
    _check(load().gdn_ssd_pool_layout_for(num_blocks, num_layers, H, P, N, G, K, act_code(act),
                                          block_align, *[ctypes.byref(o) for o in out]),
           "gdn_ssd_pool_layout_for")
    return tuple(o.value for o in out)


class Pool:
    """A state pool (gdn_state_pool_create).  With ``memory`` (a CUDA uint8
    tensor) the pool lives in that tensor, which then is a byte view of it."""

    def __init__(self, num_blocks, num_layers, Hk, Hv, dk, dv, K, act, block_align=0,
                 memory: Optional[torch.Tensor] = None):
        self.dims = (num_blocks, num_layers, Hk, Hv, dk, dv, K)
        self.act = act_code(act)
        self.num_blocks, self.num_layers = num_blocks, num_layers
        self.memory = memory
        h = ctypes.c_void_p()
        nbytes = memory.numel() * memory.element_size() if memory is not None else 0
        _check(load().gdn_state_pool_create(ctypes.byref(h), num_blocks, num_layers, Hk, Hv, dk,
                                            dv, K, self.act, block_align, _ptr(memory), nbytes),
               "gdn_state_pool_create")
        self.handle = h
        s, c, r, b = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_void_p()
        _check(load().gdn_state_pool_layout(h, ctypes.byref(s), ctypes.byref(c), ctypes.byref(r),
                                            ctypes.byref(b)), "gdn_state_pool_layout")
        self.stride, self.conv_off, self.rec_off, self.base = s.value, c.value, r.value, b.value

    def close(self):
        if self.handle is not None and self.handle.value:
            load().gdn_state_pool_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_timing_events(self, before=None, after=None):
        """Record torch.cuda.Event ``before``/``after`` around the compute
        kernels of every later forward (None, None: off)."""
        hb = before.cuda_event if before is not None else None
        ha = after.cuda_event if after is not None else None
        _check(load().gdn_pool_set_timing_events(self.handle, hb, ha),
               "gdn_pool_set_timing_events")

    def reserve(self, max_tokens: int):
        """gdn_state_pool_reserve: > 0 grow the prefill scratch now, 0 free it
        and use the fused prefill kernel only, < 0 grow on demand."""
        _check(load().gdn_state_pool_reserve(self.handle, max_tokens), "gdn_state_pool_reserve")

    def last_prefill_path(self) -> int:
        """gdn_pool_last_prefill_path: PREFILL_NONE / SPLIT / FUSED / SERIAL."""
        v = ctypes.c_int()
        _check(load().gdn_pool_last_prefill_path(self.handle, ctypes.byref(v)),
               "gdn_pool_last_prefill_path")
        return v.value

    def copy_block(self, layer, src, dst, stream=None):
        _check(load().gdn_state_pool_copy_block(self.handle, layer, src, dst, _stream(stream)),
               "gdn_state_pool_copy_block")

    def error_flags(self, layer=-1, reset=True, stream=None) -> int:
        v = ctypes.c_uint32()
        _check(load().gdn_get_error(self.handle, layer, ctypes.byref(v), 1 if reset else 0,
                                    _stream(stream)), "gdn_get_error")
        return v.value


class SsdPool(Pool):
    """A Mamba2 state pool (gdn_ssd_pool_create); ``rec_off`` is the SSM
    state's offset.  With ``memory`` the pool lives in that CUDA uint8 tensor."""

    def __init__(self, num_blocks, num_layers, H, P, N, G, K, act, block_align=0,
                 memory: Optional[torch.Tensor] = None):
        self.dims = (num_blocks, num_layers, H, P, N, G, K)
        self.act = act_code(act)
        self.num_blocks, self.num_layers = num_blocks, num_layers
        self.memory = memory
        h = ctypes.c_void_p()
        nbytes = memory.numel() * memory.element_size() if memory is not None else 0
        _check(load().gdn_ssd_pool_create(ctypes.byref(h), num_blocks, num_layers, H, P, N, G, K,
                                          self.act, block_align, _ptr(memory), nbytes),
               "gdn_ssd_pool_create")
        self.handle = h
        s, c, r, b = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_void_p()
        _check(load().gdn_state_pool_layout(h, ctypes.byref(s), ctypes.byref(c), ctypes.byref(r),
                                            ctypes.byref(b)), "gdn_state_pool_layout")
        self.stride, self.conv_off, self.rec_off, self.base = s.value, c.value, r.value, b.value


def ssd_varlen_forward(pool: SsdPool, layer: int, xbc, dt, cu_seqlens, state_block_idx, has_past,
                       conv_w, A_log, dt_bias, D, y, T: int, N: int, max_seqlen_hint: int = 0,
                       stream=None) -> None:
    """gdn_ssd_varlen_forward on device tensors (or raw device pointers)."""
    w = SsdWeights(_ptr(conv_w), _ptr(A_log), _ptr(dt_bias), _ptr(D))
    _check(load().gdn_ssd_varlen_forward(pool.handle, layer, _ptr(xbc), _ptr(dt),
                                         _ptr(cu_seqlens), _ptr(state_block_idx), _ptr(has_past),
                                         ctypes.byref(w), _ptr(y), T, N, max_seqlen_hint,
                                         _stream(stream)), "gdn_ssd_varlen_forward")


def varlen_forward(pool: Pool, layer: int, x_qkv, a, b, cu_seqlens, state_block_idx, has_past,
                   conv_w, A_log, dt_bias, out, T: int, N: int, max_seqlen_hint: int = 0,
                   stream=None) -> None:
    """gdn_varlen_forward on device tensors (or raw device pointers)."""
    w = Weights(_ptr(conv_w), _ptr(A_log), _ptr(dt_bias))
    _check(load().gdn_varlen_forward(pool.handle, layer, _ptr(x_qkv), _ptr(a), _ptr(b),
                                     _ptr(cu_seqlens), _ptr(state_block_idx), _ptr(has_past),
                                     ctypes.byref(w), _ptr(out), T, N, max_seqlen_hint,
                                     _stream(stream)), "gdn_varlen_forward")


def kda_varlen_forward(pool: Pool, layer: int, x_qkv, a, b, cu_seqlens, state_block_idx,
                       has_past, conv_w, A_log, dt_bias, out, T: int, N: int,
                       max_seqlen_hint: int = 0, stream=None) -> None:
    """gdn_kda_varlen_forward: the per-channel-decay rule (a [T][Hv][d_k],
    dt_bias [Hv][d_k]) on device tensors (or raw device pointers)."""
    w = Weights(_ptr(conv_w), _ptr(A_log), _ptr(dt_bias))
    _check(load().gdn_kda_varlen_forward(pool.handle, layer, _ptr(x_qkv), _ptr(a), _ptr(b),
                                         _ptr(cu_seqlens), _ptr(state_block_idx), _ptr(has_past),
                                         ctypes.byref(w), _ptr(out), T, N, max_seqlen_hint,
                                         _stream(stream)), "gdn_kda_varlen_forward")


def diag_umma_gemm(A, B, C, D, operand_f16=False, stream=None) -> None:
    """gdn_diag_umma_gemm: D = (C or 0) + A @ B^T on the tensor cores
    (A [128][K], B [N][K] bf16; C, D [128][N] fp32; device tensors)."""
    N, K = B.shape
    _check(load().gdn_diag_umma_gemm(_ptr(A), _ptr(B), _ptr(C), _ptr(D), N, K,
                                     1 if operand_f16 else 0, _stream(stream)),
           "gdn_diag_umma_gemm")


def diag_umma_gemm_ex(A, B, C, D, operand_f16=False, a_mn=False, b_mn=False,
                      stream=None) -> None:
    """gdn_diag_umma_gemm_ex: the same GEMM with A and/or B staged MN-major
    (a_mn=2: A in tensor memory instead)."""
    N, K = B.shape
    _check(load().gdn_diag_umma_gemm_ex(_ptr(A), _ptr(B), _ptr(C), _ptr(D), N, K,
                                        1 if operand_f16 else 0, int(a_mn),
                                        1 if b_mn else 0, _stream(stream)),
           "gdn_diag_umma_gemm_ex")


def diag_wait_timeout(flags, stream=None) -> None:
    """gdn_diag_wait_timeout: a bounded wait that runs out and ORs
    GDN_FLAG_TIMEOUT into ``flags`` (a 1-element int32/uint32 CUDA tensor)."""
    _check(load().gdn_diag_wait_timeout(_ptr(flags), _stream(stream)), "gdn_diag_wait_timeout")


def in_proj(hidden, w_qkv, w_z, w_b, w_a, x_qkv, z, b, a, C, Hv, dv, flags=None,
            stream=None) -> None:
    """gdn_in_proj: x_qkv | z | b | a = hidden W^T (device tensors)."""
    T, d_model = hidden.shape
    _check(load().gdn_in_proj(_ptr(hidden), T, d_model, _ptr(w_qkv), _ptr(w_z), _ptr(w_b),
                              _ptr(w_a), C, Hv, dv, _ptr(x_qkv), _ptr(z), _ptr(b), _ptr(a),
                              _ptr(flags), _stream(stream)), "gdn_in_proj")


def out_proj(o, z, norm_w, eps, w_out, o_norm, y, flags=None, stream=None) -> None:
    """gdn_out_proj: o_norm = gated RMS norm of o, y = o_norm W_out^T."""
    T, Hv, dv = o.shape
    d_model = w_out.shape[0]
    _check(load().gdn_out_proj(_ptr(o), _ptr(z), _ptr(norm_w), float(eps), _ptr(w_out), T, Hv,
                               dv, d_model, _ptr(o_norm), _ptr(y), _ptr(flags), _stream(stream)),
           "gdn_out_proj")


def prefill_scratch_bytes(num_blocks, Hk, Hv, dk, dv, max_tokens) -> int:
    """gdn_prefill_scratch_bytes: bytes of prefill scratch the split prefill
    needs for calls of at most max_tokens tokens."""
    out = ctypes.c_size_t(0)
    _check(load().gdn_prefill_scratch_bytes(num_blocks, Hk, Hv, dk, dv, max_tokens,
                                            ctypes.byref(out)), "gdn_prefill_scratch_bytes")
    return int(out.value)


def varlen_forward_noalloc(pool_mem, num_blocks, num_layers, Hk, Hv, dk, dv, K, act, block_align,
                           layer, x_qkv, a, b, cu_seqlens, state_block_idx, has_past, conv_w,
                           A_log, dt_bias, out, T, N, max_seqlen_hint=0, flags_out=None,
                           stream=None) -> None:
    """gdn_varlen_forward_noalloc: the forward on caller-owned pool memory
    (a CUDA uint8 tensor or a raw device pointer), allocating nothing."""
    nbytes = pool_mem.numel() * pool_mem.element_size() if hasattr(pool_mem, "numel") else 0
    w = Weights(_ptr(conv_w), _ptr(A_log), _ptr(dt_bias))
    _check(load().gdn_varlen_forward_noalloc(
        _ptr(pool_mem), nbytes, num_blocks, num_layers, Hk, Hv, dk, dv, K, act_code(act),
        block_align, layer, _ptr(x_qkv), _ptr(a), _ptr(b), _ptr(cu_seqlens),
        _ptr(state_block_idx), _ptr(has_past), ctypes.byref(w), _ptr(out), T, N,
        max_seqlen_hint, _ptr(flags_out), _stream(stream)), "gdn_varlen_forward_noalloc")
