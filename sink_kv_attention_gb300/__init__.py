"""Python binding of libsinkkv (sink + window KV attention with RoPE/YaRN on GB300).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels, reached through the C ABI declared in ``include/sinkkv.h``.  PyTorch
tensors supply device memory and the current CUDA stream.  There is no CPU
fallback: if ``libsinkkv.so`` is missing or fails to load, importing the binding's
functions raises.

C entry point          Python
sk_rope_table_*        RopeTable (+ rope_table_fill_host)
sk_rope_dynamic_*      DynamicRope (+ dynamic_factor)
sk_rope_apply          rope_apply
sk_kv_append           kv_append
sk_decode_attention    decode_attention (+ decode_workspace_bytes, decode_attention_noalloc)
sk_decode_step         decode_step (+ decode_step_workspace_bytes)
sk_prefill_attention   prefill_attention
sk_kv_rerotate         kv_rerotate
sk_kv_shift_recent     kv_shift_recent
sk_paged_*             PagedLayer, paged_append, paged_decode_attention
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsinkkv.so")

SK_OK, SK_ERR_ARG, SK_ERR_CAPACITY, SK_ERR_POSITION_RANGE, SK_ERR_UNSUPPORTED, SK_ERR_CUDA = range(6)
SK_BF16, SK_F32, SK_I8 = 0, 1, 2
SK_LAYER_RING, SK_LAYER_GLOBAL = 0, 1
SK_DEVERR_POSITION_RANGE, SK_DEVERR_CAPACITY, SK_DEVERR_TIMEOUT, SK_DEVERR_BLOCK_TABLE = 1, 2, 4, 8
SK_DEVERR_STATE = 16


class SinkKVError(RuntimeError):
    """A non-OK sk_status from the library."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {_lib().sk_status_str(status).decode()}")


class RopeConfig(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int32), ("rotary_dim", ctypes.c_int32),
                ("neox", ctypes.c_int32), ("reserved0", ctypes.c_int32),
                ("theta", ctypes.c_double), ("yarn_factor", ctypes.c_double),
                ("yarn_orig_ctx", ctypes.c_int64), ("beta_fast", ctypes.c_double),
                ("beta_slow", ctypes.c_double), ("max_positions", ctypes.c_int64)]


class KVLayerStruct(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("k_dtype", ctypes.c_int32), ("v_dtype", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("sinks", ctypes.c_int32), ("window", ctypes.c_int32), ("capacity", ctypes.c_int64),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("head", ctypes.c_void_p), ("count", ctypes.c_void_p), ("pos", ctypes.c_void_p),
                ("err", ctypes.c_void_p)]


class PagedLayerStruct(ctypes.Structure):
    _fields_ = [("k_dtype", ctypes.c_int32), ("v_dtype", ctypes.c_int32), ("batch", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("max_blocks", ctypes.c_int32), ("n_sink_blocks", ctypes.c_int32), ("sinks", ctypes.c_int32),
                ("window", ctypes.c_int32), ("n_blocks", ctypes.c_int64), ("k_pool", ctypes.c_void_p),
                ("v_pool", ctypes.c_void_p), ("block_table", ctypes.c_void_p), ("sink_block_ids", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("err", ctypes.c_void_p)]


_LIB = None

# (name, restype, argtypes) of every entry point in include/sinkkv.h
_SIGNATURES = [
    ("sk_rope_table_create", ctypes.c_int, [ctypes.POINTER(RopeConfig), ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]),
    ("sk_rope_table_rebuild", ctypes.c_int, [ctypes.c_void_p, ctypes.c_double, ctypes.c_void_p]),
    ("sk_rope_table_destroy", None, [ctypes.c_void_p]),
    ("sk_rope_table_info", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(RopeConfig), ctypes.POINTER(ctypes.c_void_p)]),
    ("sk_rope_table_fill_host", ctypes.c_int, [ctypes.POINTER(RopeConfig), ctypes.c_int32, ctypes.c_void_p]),
    ("sk_rope_dynamic_factor", ctypes.c_int, [ctypes.c_int64, ctypes.c_int64, ctypes.c_double, ctypes.c_double,
                                              ctypes.POINTER(ctypes.c_double)]),
    ("sk_rope_dynamic_create", ctypes.c_int, [ctypes.POINTER(RopeConfig), ctypes.c_double, ctypes.c_double,
                                              ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]),
    ("sk_rope_dynamic_table", ctypes.c_void_p, [ctypes.c_void_p]),
    ("sk_rope_dynamic_current_factor", ctypes.c_double, [ctypes.c_void_p]),
    ("sk_rope_dynamic_update", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.POINTER(KVLayerStruct),
                                              ctypes.c_int32, ctypes.c_void_p, ctypes.POINTER(ctypes.c_double),
                                              ctypes.POINTER(ctypes.c_int32)]),
    ("sk_rope_dynamic_destroy", None, [ctypes.c_void_p]),
    ("sk_rope_apply", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                     ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    ("sk_kv_append", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(KVLayerStruct), ctypes.c_void_p, ctypes.c_int32,
                                    ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p]),
    ("sk_decode_workspace_bytes", ctypes.c_size_t, [ctypes.POINTER(KVLayerStruct), ctypes.c_int32]),
    ("sk_decode_attention", ctypes.c_int, [ctypes.POINTER(KVLayerStruct), ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32,
                                           ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                           ctypes.c_void_p]),
    ("sk_decode_attention_noalloc", ctypes.c_int, [ctypes.POINTER(KVLayerStruct), ctypes.c_void_p, ctypes.c_int32,
                                                   ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    ("sk_decode_step_workspace_bytes", ctypes.c_size_t, [ctypes.POINTER(KVLayerStruct), ctypes.c_int32]),
    ("sk_decode_step", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(KVLayerStruct), ctypes.c_void_p, ctypes.c_int32,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    ("sk_prefill_prior_keys", ctypes.c_int64, [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]),
    ("sk_selftest_bounded_wait", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    ("sk_selftest_prefill_stall", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                                 ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32,
                                                 ctypes.c_void_p, ctypes.c_void_p]),
    ("sk_prefill_workspace_bytes", ctypes.c_size_t, [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                     ctypes.c_int64]),
    ("sk_prefill_attention", ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                            ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                            ctypes.POINTER(KVLayerStruct), ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                            ctypes.c_void_p]),
    ("sk_kv_rerotate", ctypes.c_int, [ctypes.POINTER(KVLayerStruct), ctypes.c_int32, ctypes.c_void_p,
                                      ctypes.c_void_p, ctypes.c_void_p]),
    ("sk_paged_append", ctypes.c_int, [ctypes.c_void_p, ctypes.POINTER(PagedLayerStruct), ctypes.c_void_p,
                                       ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32,
                                       ctypes.c_int32, ctypes.c_void_p]),
    ("sk_paged_decode_workspace_bytes", ctypes.c_size_t, [ctypes.POINTER(PagedLayerStruct), ctypes.c_int32]),
    ("sk_paged_decode_attention", ctypes.c_int, [ctypes.POINTER(PagedLayerStruct), ctypes.c_void_p, ctypes.c_int32,
                                                 ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                 ctypes.c_size_t, ctypes.c_void_p]),
    ("sk_kv_shift_recent", ctypes.c_int, [ctypes.POINTER(KVLayerStruct), ctypes.c_int32, ctypes.c_void_p,
                                          ctypes.c_int32, ctypes.c_void_p]),
    ("sk_sync_check", ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p,
                                     ctypes.POINTER(ctypes.c_uint32)]),
    ("sk_status_str", ctypes.c_char_p, [ctypes.c_int]),
    ("sk_version", ctypes.c_int32, []),
]

EXPORTED = [name for name, _, _ in _SIGNATURES]


def _lib():
    """Load libsinkkv.so once; raise loudly if it is missing (no fallback)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libsinkkv.so not built at {LIB_PATH}; run "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(LIB_PATH)
        for name, res, args in _SIGNATURES:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = lib
    return _LIB


def _check(status: int, what: str):
    if status != SK_OK:
        raise SinkKVError(status, what)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _sk_dtype(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return SK_BF16
    if dt == torch.float32:
        return SK_F32
    if dt == torch.int8:
        return SK_I8
    raise TypeError(f"unsupported dtype {dt}")


def _need_contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


# ---------------------------------------------------------------------------
# RoPE table
# ---------------------------------------------------------------------------

class RopeTable:
    """Library-owned cos/sin table (sk_rope_table_create / rebuild / destroy)."""

    def __init__(self, head_dim: int, rotary_dim: int, theta: float, max_positions: int,
                 neox: bool = True, yarn_factor: float = 1.0, yarn_orig_ctx: int = 4096,
                 beta_fast: float = 32.0, beta_slow: float = 1.0, stream=None):
        self.cfg = RopeConfig(head_dim, rotary_dim, 1 if neox else 0, 0, float(theta),
                              float(yarn_factor), int(yarn_orig_ctx), float(beta_fast),
                              float(beta_slow), int(max_positions))
        h = ctypes.c_void_p()
        _check(_lib().sk_rope_table_create(ctypes.byref(self.cfg), _stream(stream), ctypes.byref(h)),
               "sk_rope_table_create")
        self.handle = h

    def rebuild(self, yarn_factor: float, stream=None):
        _check(_lib().sk_rope_table_rebuild(self.handle, float(yarn_factor), _stream(stream)),
               "sk_rope_table_rebuild")
        self.cfg.yarn_factor = float(yarn_factor)

    def device_ptr(self) -> int:
        out = ctypes.c_void_p()
        _check(_lib().sk_rope_table_info(self.handle, None, ctypes.byref(out)), "sk_rope_table_info")
        return out.value

    def config(self) -> RopeConfig:
        c = RopeConfig()
        _check(_lib().sk_rope_table_info(self.handle, ctypes.byref(c), None), "sk_rope_table_info")
        return c

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            _lib().sk_rope_table_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def rope_table_fill_host(head_dim: int, rotary_dim: int, theta: float, max_positions: int, neox: bool = True,
                         yarn_factor: float = 1.0, yarn_orig_ctx: int = 4096, beta_fast: float = 32.0,
                         beta_slow: float = 1.0, n_threads: int = 0):
    """The table as sk_rope_table_fill_host builds it on the host (no device):
    numpy float32 [max_positions, rotary_dim/2, 2] of (cos, sin) pairs."""
    import numpy as np
    cfg = RopeConfig(head_dim, rotary_dim, 1 if neox else 0, 0, float(theta), float(yarn_factor),
                     int(yarn_orig_ctx), float(beta_fast), float(beta_slow), int(max_positions))
    out = np.empty((max_positions, rotary_dim // 2, 2), dtype=np.float32)
    _check(_lib().sk_rope_table_fill_host(ctypes.byref(cfg), int(n_threads), out.ctypes.data_as(ctypes.c_void_p)),
           "sk_rope_table_fill_host")
    return out


def dynamic_factor(total_positions: int, orig_ctx: int, step: float = 0.125, cap: float = 2.0) -> float:
    """The YaRN factor for a dialog of total_positions (sk_rope_dynamic_factor)."""
    f = ctypes.c_double()
    _check(_lib().sk_rope_dynamic_factor(int(total_positions), int(orig_ctx), float(step), float(cap),
                                         ctypes.byref(f)), "sk_rope_dynamic_factor")
    return f.value


class _TableView(RopeTable):
    """A table owned by another library object (not freed here)."""

    def __init__(self, handle: int, owner):
        self.handle = ctypes.c_void_p(handle)
        self._owner = owner
        self.cfg = self.config()

    def rebuild(self, yarn_factor: float, stream=None):
        raise RuntimeError("the table of a DynamicRope changes only through DynamicRope.update")

    def close(self):
        self.handle = ctypes.c_void_p()


class DynamicRope:
    """A RoPE table whose YaRN factor follows the dialog's length (sk_rope_dynamic_*).
    ``table`` is the live table to pass to kv_append / rope_apply; ``update`` picks the
    factor for a length and, on a change, turns the given layers' cached keys."""

    def __init__(self, head_dim: int, rotary_dim: int, theta: float, max_positions: int, orig_ctx: int,
                 neox: bool = True, yarn_factor: float = 1.0, beta_fast: float = 32.0, beta_slow: float = 1.0,
                 step: float = 0.125, cap: float = 0.0, stream=None):
        cfg = RopeConfig(head_dim, rotary_dim, 1 if neox else 0, 0, float(theta), float(yarn_factor),
                         int(orig_ctx), float(beta_fast), float(beta_slow), int(max_positions))
        h = ctypes.c_void_p()
        _check(_lib().sk_rope_dynamic_create(ctypes.byref(cfg), float(step), float(cap), _stream(stream),
                                             ctypes.byref(h)), "sk_rope_dynamic_create")
        self.handle = h
        self.table = _TableView(_lib().sk_rope_dynamic_table(h), self)

    @property
    def factor(self) -> float:
        return float(_lib().sk_rope_dynamic_current_factor(self.handle))

    def update(self, total_positions: int, layers: Sequence["KVLayer"] = (), stream=None):
        """Returns (factor now in force, whether it changed)."""
        arr = (KVLayerStruct * max(1, len(layers)))(*[L.struct() for L in layers])
        f = ctypes.c_double()
        sw = ctypes.c_int32()
        _check(_lib().sk_rope_dynamic_update(self.handle, int(total_positions), arr, len(layers), _stream(stream),
                                             ctypes.byref(f), ctypes.byref(sw)), "sk_rope_dynamic_update")
        return f.value, bool(sw.value)

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            self.table.close()
            _lib().sk_rope_dynamic_destroy(self.handle)
            self.handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# ---------------------------------------------------------------------------
# KV layer (caller-owned device buffers held as torch tensors)
# ---------------------------------------------------------------------------

@dataclass
class KVLayer:
    """One layer's cache for a batch, as described by sk_kv_layer.

    k, v: [batch, n_kv_heads, capacity, head_dim]; k_scale: [batch, n_kv_heads, capacity]
    float32 (int8 K only); head, count: int32 [batch] (ring); pos: int64 [batch];
    err: uint32 word as int32 [1].
    """
    kind: int
    k: torch.Tensor
    v: torch.Tensor
    pos: torch.Tensor
    sinks: int = 0
    window: int = 0
    head: Optional[torch.Tensor] = None
    count: Optional[torch.Tensor] = None
    k_scale: Optional[torch.Tensor] = None
    err: Optional[torch.Tensor] = None

    @staticmethod
    def allocate(kind: int, batch: int, n_kv_heads: int, head_dim: int, *, sinks: int = 0,
                 window: int = 0, capacity: Optional[int] = None, k_dtype=torch.bfloat16,
                 v_dtype=torch.bfloat16, device="cuda", with_v: bool = True) -> "KVLayer":
        """with_v=False leaves V as a one-row placeholder, for callers (such as a
        key rerotation) that never touch V."""
        if kind == SK_LAYER_RING:
            capacity = sinks + window
        assert capacity is not None and capacity >= 1
        k = torch.zeros(batch, n_kv_heads, capacity, head_dim, dtype=k_dtype, device=device)
        v = (torch.zeros(batch, n_kv_heads, capacity, head_dim, dtype=v_dtype, device=device) if with_v
             else torch.zeros(1, 1, 1, head_dim, dtype=v_dtype, device=device))
        ks = (torch.ones(batch, n_kv_heads, capacity, dtype=torch.float32, device=device)
              if k_dtype == torch.int8 else None)
        z32 = lambda: torch.zeros(batch, dtype=torch.int32, device=device)
        return KVLayer(kind, k, v, torch.zeros(batch, dtype=torch.int64, device=device), sinks, window,
                       z32() if kind == SK_LAYER_RING else None, z32() if kind == SK_LAYER_RING else None,
                       ks, torch.zeros(1, dtype=torch.int32, device=device))

    @property
    def batch(self):
        return self.k.shape[0]

    @property
    def n_kv_heads(self):
        return self.k.shape[1]

    @property
    def capacity(self):
        return self.k.shape[2]

    @property
    def head_dim(self):
        return self.k.shape[3]

    def struct(self) -> KVLayerStruct:
        _need_contig(self.k, self.v, self.k_scale, self.head, self.count, self.pos)
        return KVLayerStruct(self.kind, _sk_dtype(self.k.dtype), _sk_dtype(self.v.dtype), self.batch,
                             self.n_kv_heads, self.head_dim, self.sinks, self.window, self.capacity,
                             self.k.data_ptr(), self.v.data_ptr(),
                             None if self.k_scale is None else self.k_scale.data_ptr(),
                             None if self.head is None else self.head.data_ptr(),
                             None if self.count is None else self.count.data_ptr(),
                             self.pos.data_ptr(), None if self.err is None else self.err.data_ptr())

    def error_bits(self) -> int:
        """Read the device error word (synchronises)."""
        return 0 if self.err is None else int(self.err.item()) & 0xFFFFFFFF


# ---------------------------------------------------------------------------
# Entry points
# ---------------------------------------------------------------------------

def rope_apply(table: RopeTable, x: torch.Tensor, positions: torch.Tensor,
               err: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Rotate x [n_tok, H, D] in place at positions [n_tok] (sk_rope_apply)."""
    _need_contig(x, positions)
    n_tok, H = x.shape[0], x.shape[1]
    _check(_lib().sk_rope_apply(table.handle, _ptr(x), _sk_dtype(x.dtype), n_tok, H, _ptr(positions),
                                _ptr(err), _stream(stream)), "sk_rope_apply")
    return x


def kv_append(table: Optional[RopeTable], layer: KVLayer, q: Optional[torch.Tensor], k: torch.Tensor,
              v: torch.Tensor, stream=None):
    """Fused RoPE + append of T tokens per sequence (sk_kv_append).

    q [B, T, Hq, D] (optional) and k [B, T, Hkv, D] are rotated in place; v [B, T, Hkv, D].
    table None: k is already rotated and is appended as given (q must be None)."""
    _need_contig(q, k, v)
    T = k.shape[1]
    hq = 0 if q is None else q.shape[2]
    s = layer.struct()
    _check(_lib().sk_kv_append(None if table is None else table.handle, ctypes.byref(s), _ptr(q), hq, _ptr(k),
                               _ptr(v),
                               _sk_dtype(k.dtype), T, _stream(stream)), "sk_kv_append")


def decode_workspace_bytes(layer: KVLayer, n_q_heads: int) -> int:
    s = layer.struct()
    return int(_lib().sk_decode_workspace_bytes(ctypes.byref(s), n_q_heads))


def _sink_logits(sink_logits: Optional[torch.Tensor], n_q_heads: int):
    """Checks learned sink logits (float32 [n_q_heads] on the device, or None)."""
    if sink_logits is None:
        return None
    if sink_logits.dtype != torch.float32 or sink_logits.numel() != n_q_heads or not sink_logits.is_contiguous():
        raise ValueError("sink_logits must be a contiguous float32 tensor of n_q_heads values")
    return _ptr(sink_logits)


def decode_attention(layer: KVLayer, q_rot: torch.Tensor, out: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None, stream=None,
                     sink_logits: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Split-K decode attention of q_rot [B, Hq, D] over the layer's visible set;
    optional learned per-head sink logits (float32 [Hq], clamped to [-10, 15])."""
    _need_contig(q_rot)
    Hq = q_rot.shape[1]
    if out is None:
        out = torch.empty_like(q_rot)
    s = layer.struct()
    need = int(_lib().sk_decode_workspace_bytes(ctypes.byref(s), Hq))
    if need == 0:
        raise SinkKVError(SK_ERR_UNSUPPORTED, "sk_decode_workspace_bytes")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_rot.device)
    _check(_lib().sk_decode_attention(ctypes.byref(s), _ptr(q_rot), Hq, _sk_dtype(q_rot.dtype),
                                      _sink_logits(sink_logits, Hq), _ptr(out), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream)),
           "sk_decode_attention")
    return out


def decode_attention_noalloc(layer: KVLayer, q_rot: torch.Tensor, out: torch.Tensor, stream=None,
                             sink_logits: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Decode attention for callers that cannot allocate device memory: the scratch
    is the library's fixed 4 MiB device array (sk_decode_attention_noalloc); `out`
    must be given.  Calls that may overlap on the GPU race on that array."""
    _need_contig(q_rot, out)
    s = layer.struct()
    _check(_lib().sk_decode_attention_noalloc(ctypes.byref(s), _ptr(q_rot), q_rot.shape[1],
                                              _sk_dtype(q_rot.dtype), _sink_logits(sink_logits, q_rot.shape[1]),
                                              _ptr(out), _stream(stream)),
           "sk_decode_attention_noalloc")
    return out


def decode_step_workspace_bytes(layer: KVLayer, n_q_heads: int) -> int:
    s = layer.struct()
    return int(_lib().sk_decode_step_workspace_bytes(ctypes.byref(s), n_q_heads))


def decode_step(table: Optional[RopeTable], layer: KVLayer, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None, stream=None,
                sink_logits: Optional[torch.Tensor] = None) -> torch.Tensor:
    """One decode token per sequence: RoPE + append + attention in two kernels
    (sk_decode_step).  q [B, Hq, D], k and v [B, Hkv, D], unrotated and left as they are
    (unlike kv_append); returns out [B, Hq, D].  table None: q and k come rotated."""
    _need_contig(q, k, v)
    Hq = q.shape[1]
    if out is None:
        out = torch.empty_like(q)
    s = layer.struct()
    need = int(_lib().sk_decode_step_workspace_bytes(ctypes.byref(s), Hq))
    if need == 0:
        raise SinkKVError(SK_ERR_UNSUPPORTED, "sk_decode_step_workspace_bytes")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(_lib().sk_decode_step(None if table is None else table.handle, ctypes.byref(s), _ptr(q), Hq, _ptr(k),
                                 _ptr(v), _sk_dtype(q.dtype), _sink_logits(sink_logits, Hq), _ptr(out),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)),
           "sk_decode_step")
    return out


def prefill_prior_keys(p0: int, sinks: int, window: int) -> int:
    """Keys a chunk starting at p0 takes from a prior cache (sk_prefill_prior_keys)."""
    n = int(_lib().sk_prefill_prior_keys(int(p0), int(sinks), int(window)))
    if n < 0:
        raise SinkKVError(SK_ERR_ARG, "sk_prefill_prior_keys")
    return n


def prefill_workspace_bytes(batch: int, T: int, n_kv_heads: int, head_dim: int, prior_keys: int = 0) -> int:
    return int(_lib().sk_prefill_workspace_bytes(batch, T, n_kv_heads, head_dim, int(prior_keys)))


def prefill_attention(q_rot: torch.Tensor, k_rot: torch.Tensor, v: torch.Tensor, p0: int, sinks: int,
                      window: int, out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                      err: Optional[torch.Tensor] = None, stream=None,
                      sink_logits: Optional[torch.Tensor] = None,
                      prior: Optional["KVLayer"] = None) -> torch.Tensor:
    """Masked prefill attention of a chunk: q [B,T,Hq,D], k/v [B,T,Hkv,D]
    (sk_prefill_attention); window <= 0 is a global layer; optional learned per-head
    sink logits (float32 [Hq]); ``prior``: the layer whose cache holds positions
    [0, p0) of every sequence (the chunk not yet appended), whose keys the chunk then
    also sees."""
    _need_contig(q_rot, k_rot, v)
    B, T, Hq, D = q_rot.shape
    Hkv = k_rot.shape[2]
    if out is None:
        out = torch.empty_like(q_rot)
    prior_keys = prefill_prior_keys(p0, sinks, window) if prior is not None else 0
    need = prefill_workspace_bytes(B, T, Hkv, D, prior_keys)
    if need == 0:
        raise SinkKVError(SK_ERR_UNSUPPORTED, "sk_prefill_workspace_bytes")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_rot.device)
    ps = ctypes.byref(prior.struct()) if prior is not None else None
    _check(_lib().sk_prefill_attention(_ptr(q_rot), _ptr(k_rot), _ptr(v), B, T, Hq, Hkv, D, int(p0), int(sinks),
                                       int(window), ps, _sink_logits(sink_logits, Hq), _ptr(out), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _ptr(err), _stream(stream)),
           "sk_prefill_attention")
    return out


def kv_rerotate(layers: Sequence[KVLayer], table_from: RopeTable, table_to: RopeTable, stream=None):
    """Turn every cached key of `layers` from table_from's factor to table_to's (sk_kv_rerotate)."""
    arr = (KVLayerStruct * len(layers))(*[l.struct() for l in layers])
    _check(_lib().sk_kv_rerotate(arr, len(layers), table_from.handle, table_to.handle, _stream(stream)),
           "sk_kv_rerotate")


@dataclass
class PagedLayer:
    """A paged layer's caller-owned device buffers (sk_paged_layer): pools
    [n_blocks, H_kv, block_size, D], block_table int32 [B, max_blocks] (-1 = no block),
    sink_block_ids int32 [n_sink_blocks], seq_lens int64 [B]."""
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    block_table: torch.Tensor
    sink_block_ids: Optional[torch.Tensor]
    seq_lens: torch.Tensor
    err: torch.Tensor
    sinks: int
    window: int

    @staticmethod
    def allocate(batch: int, n_kv_heads: int, head_dim: int, *, block_size: int, n_blocks: int, max_blocks: int,
                 sinks: int = 0, window: int = 0, n_sink_blocks: int = 0, dtype=torch.bfloat16,
                 device="cuda") -> "PagedLayer":
        z = dict(dtype=dtype, device=device)
        return PagedLayer(
            k_pool=torch.zeros(n_blocks, n_kv_heads, block_size, head_dim, **z),
            v_pool=torch.zeros(n_blocks, n_kv_heads, block_size, head_dim, **z),
            block_table=torch.full((batch, max_blocks), -1, dtype=torch.int32, device=device),
            sink_block_ids=(torch.arange(n_sink_blocks, dtype=torch.int32, device=device)
                            if n_sink_blocks > 0 else None),
            seq_lens=torch.zeros(batch, dtype=torch.int64, device=device),
            err=torch.zeros(1, dtype=torch.int32, device=device), sinks=sinks, window=window)

    @property
    def batch(self):
        return self.block_table.shape[0]

    @property
    def n_kv_heads(self):
        return self.k_pool.shape[1]

    @property
    def block_size(self):
        return self.k_pool.shape[2]

    def struct(self) -> PagedLayerStruct:
        n_sink = 0 if self.sink_block_ids is None else self.sink_block_ids.numel()
        return PagedLayerStruct(_sk_dtype(self.k_pool.dtype), _sk_dtype(self.v_pool.dtype), self.batch,
                                self.n_kv_heads, self.k_pool.shape[3], self.block_size, self.block_table.shape[1],
                                n_sink, self.sinks, self.window, self.k_pool.shape[0], self.k_pool.data_ptr(),
                                self.v_pool.data_ptr(), self.block_table.data_ptr(),
                                None if self.sink_block_ids is None else self.sink_block_ids.data_ptr(),
                                self.seq_lens.data_ptr(), self.err.data_ptr())

    def error_bits(self) -> int:
        return int(self.err.item())


def paged_append(table: RopeTable, layer: PagedLayer, q: Optional[torch.Tensor], k: torch.Tensor, v: torch.Tensor,
                 stream=None):
    """RoPE on q (optional) and k in place, then k, v into the pool slots of the block
    table (sk_paged_append); q [B, T, Hq, D], k/v [B, T, Hkv, D]."""
    _need_contig(k, v)
    if q is not None:
        _need_contig(q)
    s = layer.struct()
    _check(_lib().sk_paged_append(table.handle, ctypes.byref(s), _ptr(q), 0 if q is None else q.shape[2], _ptr(k),
                                  _ptr(v), _sk_dtype(k.dtype), k.shape[1], _stream(stream)), "sk_paged_append")


def paged_decode_workspace_bytes(layer: PagedLayer, n_q_heads: int) -> int:
    s = layer.struct()
    return int(_lib().sk_paged_decode_workspace_bytes(ctypes.byref(s), n_q_heads))


def paged_decode_attention(layer: PagedLayer, q_rot: torch.Tensor, out: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None, stream=None,
                           sink_logits: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Decode attention of q_rot [B, Hq, D] over a paged layer (sk_paged_decode_attention)."""
    _need_contig(q_rot)
    Hq = q_rot.shape[1]
    if out is None:
        out = torch.empty_like(q_rot)
    s = layer.struct()
    need = int(_lib().sk_paged_decode_workspace_bytes(ctypes.byref(s), Hq))
    if need == 0:
        raise SinkKVError(SK_ERR_UNSUPPORTED, "sk_paged_decode_workspace_bytes")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=q_rot.device)
    _check(_lib().sk_paged_decode_attention(ctypes.byref(s), _ptr(q_rot), Hq, _sk_dtype(q_rot.dtype),
                                            _sink_logits(sink_logits, Hq), _ptr(out), _ptr(workspace),
                                            workspace.numel() * workspace.element_size(), _stream(stream)),
           "sk_paged_decode_attention")
    return out


def kv_shift_recent(layers: Sequence[KVLayer], table: RopeTable, delta: int, stream=None):
    """Turn the recent keys of ring layers by `delta` positions in place; sinks and
    values stay (sk_kv_shift_recent)."""
    arr = (KVLayerStruct * max(1, len(layers)))(*[L.struct() for L in layers])
    _check(_lib().sk_kv_shift_recent(arr, len(layers), table.handle, int(delta), _stream(stream)),
           "sk_kv_shift_recent")


def sync_check(err: torch.Tensor, clear: bool = False, stream=None):
    """(status, bits) of a device error word after the queued work (sk_sync_check)."""
    bits = ctypes.c_uint32()
    st = _lib().sk_sync_check(_ptr(err), 1 if clear else 0, _stream(stream), ctypes.byref(bits))
    return int(st), int(bits.value)


def selftest_bounded_wait(err: torch.Tensor, stream=None) -> None:
    """Launch the bounded-wait diagnostic (sk_selftest_bounded_wait): about one second
    later SK_DEVERR_TIMEOUT is set in `err`."""
    _check(_lib().sk_selftest_bounded_wait(_ptr(err), _stream(stream)), "sk_selftest_bounded_wait")


def selftest_prefill_stall(q_rot: torch.Tensor, k_rot: torch.Tensor, v: torch.Tensor, stall_tile: int,
                           err: torch.Tensor, stream=None) -> torch.Tensor:
    """Run the prefill pipeline on a global causal chunk whose P of tile `stall_tile` is
    never signalled ready (sk_selftest_prefill_stall): the blocks that reach it give up
    after about one second and set SK_DEVERR_TIMEOUT in `err`.  Returns the (undefined)
    output buffer."""
    _need_contig(q_rot, k_rot, v)
    B, T, Hq, D = q_rot.shape
    Hkv = k_rot.shape[2]
    out = torch.empty_like(q_rot)
    need = prefill_workspace_bytes(B, T, Hkv, D, 0)
    if need == 0:
        raise SinkKVError(SK_ERR_UNSUPPORTED, "sk_prefill_workspace_bytes")
    ws = torch.empty(need, dtype=torch.uint8, device=q_rot.device)
    _check(_lib().sk_selftest_prefill_stall(_ptr(q_rot), _ptr(k_rot), _ptr(v), B, T, Hq, Hkv, D, _ptr(out), _ptr(ws),
                                            need, int(stall_tile), _ptr(err), _stream(stream)),
           "sk_selftest_prefill_stall")
    return out


def version() -> int:
    return int(_lib().sk_version())
