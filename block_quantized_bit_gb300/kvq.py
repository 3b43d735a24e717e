"""Thin ctypes binding of libkvq (``include/kvq.h``), with the same entry-point names.

Argument marshalling only: torch tensors are passed as raw device pointers plus sizes, and the
current torch CUDA stream as the ``stream`` argument.  Every step of the store and the decode runs
in libkvq's CUDA kernels.  If the library has not been built, importing works but every call raises
``RuntimeError`` -- there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkvq.so")

KVQ_FP8_E4M3 = 1
KVQ_Q8_0 = 2
KVQ_FP8_E4M3_UNSCALED = 3
KVQ_FP8_E5M2_UNSCALED = 4
KIND = {"fp8_e4m3": KVQ_FP8_E4M3, "q8_0": KVQ_Q8_0, "fp8_e4m3_unscaled": KVQ_FP8_E4M3_UNSCALED,
        "fp8_e5m2_unscaled": KVQ_FP8_E5M2_UNSCALED}
KVQ_OUT_BF16 = 0
KVQ_OUT_F32 = 1

STATUS = {0: "KVQ_OK", -1: "KVQ_EINVAL", -2: "KVQ_EKIND", -3: "KVQ_EHEADDIM", -4: "KVQ_EALIGN",
          -5: "KVQ_EWORKSPACE", -6: "KVQ_EARCH", -7: "KVQ_ECUDA", -8: "KVQ_EUNSUPPORTED", -9: "KVQ_ETIMEOUT"}

EXPORTS = ["kvq_pool_bytes", "kvq_scale_bytes", "kvq_bytes_per_token", "kvq_num_pages", "kvq_store",
           "kvq_decode_workspace_bytes", "kvq_decode_workspace_bytes_ex", "kvq_decode_path",
           "kvq_decode_sparse_workspace_bytes", "kvq_decode_sparse", "kvq_decode", "kvq_decode_ex",
           "kvq_workspace_status", "kvq_encode_probe", "kvq_quantize_probe", "kvq_dequant_probe", "kvq_strerror",
           "kvq_device_check", "kvq_version", "kvq_decode_noalloc", "kvq_noalloc_status", "kvq_wait_probe",
           "kvq_extend_workspace_bytes", "kvq_extend", "kvq_store_act_quant", "kvq_store_unscaled",
           "kvq_bytes_per_token_ex", "kvq_num_pages_ex", "kvq_exp2_probe", "kvq_extend_workspace_bytes_ex",
           "kvq_extend_ex", "kvq_extend_path"]


class kvq_layout(ctypes.Structure):
    _fields_ = [("num_pages", ctypes.c_int64), ("page_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("v_dim", ctypes.c_int32), ("mla", ctypes.c_int32)]


class kvq_decode_options(ctypes.Structure):
    _fields_ = [("pages_per_split", ctypes.c_int32), ("path", ctypes.c_int32)]


class kvq_extend_options(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int32), ("precise_p", ctypes.c_int32)]


class KvqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s failed: %s (%s)" % (where, STATUS.get(status, status), strerror(status)))


_lib = None


def lib():
    """The loaded libkvq (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libkvq.so is not built (%s); run __graft_entry__.build()" % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_size_t
        LP = ctypes.POINTER(kvq_layout)
        OP = ctypes.POINTER(kvq_decode_options)
        EP = ctypes.POINTER(kvq_extend_options)
        sig = {
            "kvq_pool_bytes": (sz, [LP]),
            "kvq_scale_bytes": (sz, [LP]),
            "kvq_bytes_per_token": (ctypes.c_double, [LP]),
            "kvq_num_pages": (i64, [LP, sz]),
            "kvq_bytes_per_token_ex": (ctypes.c_double, [LP, i32]),
            "kvq_num_pages_ex": (i64, [LP, i32, sz]),
            "kvq_store": (i32, [P, P, P, P, P, i64, LP, i32, P]),
            "kvq_decode_workspace_bytes": (sz, [LP, i32, i32, i32]),
            "kvq_decode_workspace_bytes_ex": (sz, [LP, i32, i32, i32, OP]),
            "kvq_decode_path": (i32, [LP, i32, i32, i32, OP]),
            "kvq_decode_sparse_workspace_bytes": (sz, [LP, i32, i32, i32]),
            "kvq_decode_sparse": (i32, [P, P, P, P, i32, P, P, i32, i32, i32, ctypes.c_float, P, i32, P, sz, LP,
                                        i32, P]),
            "kvq_decode": (i32, [P, P, P, P, i32, P, i32, i32, ctypes.c_float, P, i32, P, sz, LP, i32, P]),
            "kvq_extend_workspace_bytes": (sz, []),
            "kvq_store_act_quant": (i32, [P, P, P, P, i64, i32, LP, i32, P]),
            "kvq_store_unscaled": (i32, [P, P, P, P, i64, LP, i32, P]),
            "kvq_extend": (i32, [P, P, P, P, i32, P, P, i32, i32, i32, ctypes.c_float, P, i32, P, sz, LP, i32, P]),
            "kvq_decode_ex": (i32, [P, P, P, P, i32, P, i32, i32, ctypes.c_float, P, i32, P, sz, LP, i32, OP, P]),
            "kvq_workspace_status": (i32, [P, P]),
            "kvq_encode_probe": (i32, [i32, P, P, i64, P]),
            "kvq_dequant_probe": (i32, [i32, P, P, P, i64, P]),
            "kvq_quantize_probe": (i32, [i32, P, i64, P, i64, P, P]),
            "kvq_strerror": (ctypes.c_char_p, [i32]),
            "kvq_device_check": (i32, []),
            "kvq_version": (ctypes.c_char_p, []),
            "kvq_decode_noalloc": (i32, [P, P, P, P, i32, P, i32, i32, ctypes.c_float, P, i32, LP, i32, P]),
            "kvq_wait_probe": (i32, [P, P]),
            "kvq_noalloc_status": (i32, [P]),
            "kvq_exp2_probe": (i32, [P, P, i64, P]),
            "kvq_extend_workspace_bytes_ex": (sz, [LP, i32, i32, i32, EP]),
            "kvq_extend_path": (i32, [LP, i32, i32, i32, EP]),
            "kvq_extend_ex": (i32, [P, P, P, P, i32, P, P, i32, i32, i32, ctypes.c_float, P, i32, P, sz, LP, i32,
                                    EP, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def strerror(status: int) -> str:
    return lib().kvq_strerror(int(status)).decode()


def _check(status: int, where: str):
    if status != 0:
        raise KvqError(status, where)


def _kind(kind) -> int:
    return KIND[kind] if isinstance(kind, str) else int(kind)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


@dataclass
class Layout:
    """Python view of ``kvq_layout``."""
    num_pages: int
    page_size: int
    num_kv_heads: int
    head_dim: int
    v_dim: int
    mla: bool = False

    def c(self) -> kvq_layout:
        return kvq_layout(self.num_pages, self.page_size, self.num_kv_heads, self.head_dim, self.v_dim,
                          int(bool(self.mla)))

    @property
    def n_kv(self) -> int:
        return 1 if self.mla else 2

    def codes_shape(self):
        return (self.num_pages, self.n_kv, self.num_kv_heads, self.page_size, self.head_dim)

    def scales_shape(self):
        return (self.num_pages, self.n_kv, self.num_kv_heads, self.page_size, self.head_dim // 32)


# ---------------------------------------------------------------------------- cost model
def kvq_pool_bytes(layout: Layout) -> int:
    return lib().kvq_pool_bytes(ctypes.byref(layout.c()))


def kvq_scale_bytes(layout: Layout) -> int:
    return lib().kvq_scale_bytes(ctypes.byref(layout.c()))


def kvq_bytes_per_token(layout: Layout) -> float:
    return lib().kvq_bytes_per_token(ctypes.byref(layout.c()))


def kvq_num_pages(layout: Layout, budget_bytes: int) -> int:
    return lib().kvq_num_pages(ctypes.byref(layout.c()), int(budget_bytes))


def kvq_bytes_per_token_ex(layout: Layout, kind) -> float:
    return lib().kvq_bytes_per_token_ex(ctypes.byref(layout.c()), _kind(kind))


def kvq_num_pages_ex(layout: Layout, kind, budget_bytes: int) -> int:
    return lib().kvq_num_pages_ex(ctypes.byref(layout.c()), _kind(kind), int(budget_bytes))


def alloc_pool(layout: Layout, device="cuda"):
    """(codes uint8, scales as int16 bit patterns) tensors of the pool's shapes on ``device``."""
    codes = torch.empty(layout.codes_shape(), dtype=torch.uint8, device=device)
    scales = torch.empty(layout.scales_shape(), dtype=torch.int16, device=device)
    return codes, scales


# ---------------------------------------------------------------------------- store
def kvq_store(pool: torch.Tensor, scales: torch.Tensor, k: torch.Tensor, v: Optional[torch.Tensor],
              slot_mapping: torch.Tensor, layout: Layout, kind, stream=None):
    """Quantize rows ``k`` / ``v`` ([T, Hkv, D] bf16) and scatter them to ``slot_mapping`` ([T] int64)."""
    _check(lib().kvq_store(_ptr(pool), _ptr(scales), _ptr(k), _ptr(v), _ptr(slot_mapping), int(k.shape[0]),
                           ctypes.byref(layout.c()), _kind(kind), _stream(stream)), "kvq_store")


# ---------------------------------------------------------------------------- decode
def _opts(pages_per_split=0, path=0):
    return kvq_decode_options(int(pages_per_split), int(path))


def kvq_decode_workspace_bytes(layout: Layout, batch: int, num_q_heads: int, max_pages_per_seq: int,
                               pages_per_split=0, path=0) -> int:
    o = _opts(pages_per_split, path)
    return lib().kvq_decode_workspace_bytes_ex(ctypes.byref(layout.c()), int(batch), int(num_q_heads),
                                               int(max_pages_per_seq), ctypes.byref(o))


def kvq_decode_path(layout: Layout, batch: int, num_q_heads: int, max_pages_per_seq: int, pages_per_split=0,
                    path=0) -> int:
    """1 (CUDA cores, one launch) or 2 (tensor cores + merge, two launches); negative status if none."""
    o = _opts(pages_per_split, path)
    return lib().kvq_decode_path(ctypes.byref(layout.c()), int(batch), int(num_q_heads), int(max_pages_per_seq),
                                 ctypes.byref(o))


def alloc_workspace(layout: Layout, batch, num_q_heads, max_pages_per_seq, device="cuda", **opts):
    n = kvq_decode_workspace_bytes(layout, batch, num_q_heads, max_pages_per_seq, **opts)
    if n == 0:
        raise KvqError(-1, "kvq_decode_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def kvq_decode(q: torch.Tensor, pool: torch.Tensor, scales: torch.Tensor, block_table: torch.Tensor,
               seq_lens: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor, layout: Layout, kind,
               sm_scale: float = 1.0, pages_per_split: int = 0, path: int = 0, stream=None):
    """Decode attention; writes ``out`` ([B, Hq, v_dim], bf16 or float32)."""
    if out.dtype == torch.bfloat16:
        od = KVQ_OUT_BF16
    elif out.dtype == torch.float32:
        od = KVQ_OUT_F32
    else:
        raise TypeError("out must be bfloat16 or float32")
    o = _opts(pages_per_split, path)
    _check(lib().kvq_decode_ex(_ptr(q), _ptr(pool), _ptr(scales), _ptr(block_table), int(block_table.shape[1]),
                               _ptr(seq_lens), int(seq_lens.shape[0]), int(q.shape[1]), float(sm_scale), _ptr(out),
                               od, _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                               ctypes.byref(layout.c()), _kind(kind), ctypes.byref(o), _stream(stream)),
           "kvq_decode")


def kvq_decode_noalloc(q: torch.Tensor, pool: torch.Tensor, scales: torch.Tensor, block_table: torch.Tensor,
                       seq_lens: torch.Tensor, out: torch.Tensor, layout: Layout, kind, sm_scale: float = 1.0,
                       stream=None):
    """kvq_decode without a workspace argument, for callers that cannot allocate device memory.

    The split-K scratch is the library's fixed device array (KVQ_NOALLOC_SCRATCH_BYTES); calls that
    overlap on the GPU share it and race.
    """
    od = KVQ_OUT_BF16 if out.dtype == torch.bfloat16 else KVQ_OUT_F32
    _check(lib().kvq_decode_noalloc(_ptr(q), _ptr(pool), _ptr(scales), _ptr(block_table), int(block_table.shape[1]),
                                    _ptr(seq_lens), int(seq_lens.shape[0]), int(q.shape[1]), float(sm_scale),
                                    _ptr(out), od, ctypes.byref(layout.c()), _kind(kind), _stream(stream)),
           "kvq_decode_noalloc")


def alloc_sparse_workspace(layout: Layout, batch: int, num_q_heads: int, topk: int, device="cuda"):
    n = lib().kvq_decode_sparse_workspace_bytes(ctypes.byref(layout.c()), int(batch), int(num_q_heads), int(topk))
    if n == 0:
        raise KvqError(-1, "kvq_decode_sparse_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def kvq_decode_sparse(q: torch.Tensor, pool: torch.Tensor, scales: torch.Tensor, block_table: torch.Tensor,
                      seq_lens: torch.Tensor, indices: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
                      layout: Layout, kind, sm_scale: float = 1.0, stream=None):
    """Sparse (top-K) decode over the columns ``indices`` ([B, topk] int32, -1 = masked) selects."""
    if out.dtype == torch.bfloat16:
        od = KVQ_OUT_BF16
    elif out.dtype == torch.float32:
        od = KVQ_OUT_F32
    else:
        raise TypeError("out must be bfloat16 or float32")
    B, Hq = q.shape[0], q.shape[1]
    topk = indices.shape[1] if indices.dim() == 2 else 0
    _check(lib().kvq_decode_sparse(_ptr(q), _ptr(pool), _ptr(scales), _ptr(block_table), int(block_table.shape[1]),
                                   _ptr(seq_lens), _ptr(indices), int(topk), int(B), int(Hq), float(sm_scale),
                                   _ptr(out), od, _ptr(workspace), int(workspace.numel() * workspace.element_size()),
                                   ctypes.byref(layout.c()),
                                   _kind(kind), _stream(stream)), "kvq_decode_sparse")


def kvq_store_unscaled(pool: torch.Tensor, k: torch.Tensor, v, slot_mapping: torch.Tensor, layout: Layout, kind,
                       stream=None):
    """Store into an unscaled fp8 pool (kind "fp8_e4m3_unscaled" or "fp8_e5m2_unscaled"): the plain cast."""
    _check(lib().kvq_store_unscaled(_ptr(pool), _ptr(k), None if v is None else _ptr(v), _ptr(slot_mapping),
                                    int(k.shape[0]), ctypes.byref(layout.c()), _kind(kind), _stream(stream)),
           "kvq_store_unscaled")


def kvq_store_act_quant(pool: torch.Tensor, scales: torch.Tensor, kv: torch.Tensor, slot_mapping: torch.Tensor,
                        layout: Layout, kind, rope_dim: int = 64, stream=None):
    """The MLA store fused with the model's per-64 E4M3 rounding of the latent: kv is bf16 [T, head_dim]."""
    _check(lib().kvq_store_act_quant(_ptr(pool), _ptr(scales), _ptr(kv), _ptr(slot_mapping), int(kv.shape[0]),
                                     int(rope_dim), ctypes.byref(layout.c()), _kind(kind), _stream(stream)),
           "kvq_store_act_quant")


def _extend_opts(path, precise_p=False):
    if path is None and not precise_p:
        return None
    return ctypes.byref(kvq_extend_options(int(path or 0), 1 if precise_p else 0))


def alloc_extend_workspace(device="cuda", layout: Optional[Layout] = None, total_q=0, num_q_heads=1,
                           max_pages_per_seq=1, path=None, precise_p=False):
    """The extend's workspace for these sizes and kernel choice (path None or 0: automatic; 1: each new
    token's prefix on the CUDA-core decode; 2: the flash kernel / the MLA tensor-core decode; precise_p: P
    carried to 16 bits or more).  Without a layout: the flash kernel's status word."""
    if layout is None:
        n = lib().kvq_extend_workspace_bytes()
    else:
        n = lib().kvq_extend_workspace_bytes_ex(ctypes.byref(layout.c()), int(total_q), int(num_q_heads),
                                                int(max_pages_per_seq), _extend_opts(path, precise_p))
        if n == 0:
            raise KvqError(-1, "kvq_extend_workspace_bytes_ex")
    return torch.empty(n, dtype=torch.uint8, device=device)


def kvq_extend_path(layout: Layout, total_q, num_q_heads, max_pages_per_seq, path=None, precise_p=False) -> int:
    """3 (flash kernel), 4 (flash, P as two bf16 terms), 1 or 2 (prefixes on the CUDA-core / tensor-core
    decode), or a negative status."""
    return lib().kvq_extend_path(ctypes.byref(layout.c()), int(total_q), int(num_q_heads), int(max_pages_per_seq),
                                 _extend_opts(path, precise_p))


def kvq_extend(q: torch.Tensor, pool: torch.Tensor, scales: torch.Tensor, block_table: torch.Tensor,
               seq_lens: torch.Tensor, q_start: torch.Tensor, out: torch.Tensor, workspace: torch.Tensor,
               layout: Layout, kind, sm_scale: float = 1.0, stream=None, path=None, precise_p=False):
    """Extend (prefill) attention: the q rows q_start[b] .. q_start[b+1]-1 ([total_q, Hq, D] bf16) are the
    last new tokens of sequence b and attend causally over the pool; out is [total_q, Hq, Dv].  path None
    (and no precise_p) calls kvq_extend (automatic), else kvq_extend_ex with those options."""
    if out.dtype == torch.bfloat16:
        od = KVQ_OUT_BF16
    elif out.dtype == torch.float32:
        od = KVQ_OUT_F32
    else:
        raise TypeError("out must be bfloat16 or float32")
    total_q, Hq = q.shape[0], q.shape[1]
    B = seq_lens.numel()
    args = (_ptr(q), _ptr(pool), _ptr(scales), _ptr(block_table), int(block_table.shape[1]), _ptr(seq_lens),
            _ptr(q_start), int(total_q), int(B), int(Hq), float(sm_scale), _ptr(out), od, _ptr(workspace),
            int(workspace.numel() * workspace.element_size()), ctypes.byref(layout.c()), _kind(kind))
    opts = _extend_opts(path, precise_p)
    if opts is None:
        _check(lib().kvq_extend(*args, _stream(stream)), "kvq_extend")
    else:
        _check(lib().kvq_extend_ex(*args, opts, _stream(stream)), "kvq_extend_ex")


def kvq_workspace_status(workspace: torch.Tensor, stream=None) -> int:
    return lib().kvq_workspace_status(_ptr(workspace), _stream(stream))


def kvq_noalloc_status(stream=None) -> int:
    """Status word the last kvq_decode_noalloc left in the library's scratch (0 = KVQ_OK)."""
    return lib().kvq_noalloc_status(_stream(stream))


# ---------------------------------------------------------------------------- probes
def kvq_encode_probe(kind, y: torch.Tensor, codes: torch.Tensor, stream=None):
    _check(lib().kvq_encode_probe(_kind(kind), _ptr(y), _ptr(codes), int(y.numel()), _stream(stream)),
           "kvq_encode_probe")


def kvq_quantize_probe(kind, x_bits: torch.Tensor, s_bits: torch.Tensor, codes: torch.Tensor, stream=None):
    """codes[i * nx + j] = the store's code of bf16 x[j] against nonzero fp16 scale s[i]."""
    _check(lib().kvq_quantize_probe(_kind(kind), _ptr(x_bits), int(x_bits.numel()), _ptr(s_bits), int(s_bits.numel()),
                                    _ptr(codes), _stream(stream)), "kvq_quantize_probe")


def kvq_dequant_probe(kind, codes: torch.Tensor, scales: torch.Tensor, out: torch.Tensor, stream=None):
    _check(lib().kvq_dequant_probe(_kind(kind), _ptr(codes), _ptr(scales), _ptr(out), int(codes.numel()),
                                   _stream(stream)), "kvq_dequant_probe")


def kvq_exp2_probe(x: torch.Tensor, y: torch.Tensor, stream=None):
    """y = 2^x by the extend kernel's FMA-pipe exponential (float32 device tensors of equal size)."""
    _check(lib().kvq_exp2_probe(_ptr(x), _ptr(y), int(x.numel()), _stream(stream)), "kvq_exp2_probe")


def kvq_wait_probe(workspace: torch.Tensor, stream=None):
    """One bounded wait that never completes: afterwards kvq_workspace_status(workspace) is KVQ_ETIMEOUT."""
    _check(lib().kvq_wait_probe(_ptr(workspace), _stream(stream)), "kvq_wait_probe")


def kvq_device_check() -> int:
    return lib().kvq_device_check()


def kvq_version() -> str:
    return lib().kvq_version().decode()
