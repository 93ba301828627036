"""Thin Python binding of libpic (include/pic.h): ctypes marshalling only.

Every function keeps its C name.  Device buffers are torch tensors (their
``data_ptr()`` and strides are passed through); the stream is torch's current
CUDA stream unless one is given.  Every step of the path runs in libpic's
kernels; nothing here computes.  A missing or unloadable libpic raises
immediately -- there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

from . import _build

PIC_OK = 0
STATUS_NAMES = {
    0: "PIC_OK", 1: "PIC_ERR_INVALID_ARG", 2: "PIC_ERR_UNKNOWN_CHUNK", 3: "PIC_ERR_KEY_CONFLICT",
    4: "PIC_ERR_OUT_OF_BLOCKS", 5: "PIC_ERR_CAPACITY", 6: "PIC_ERR_RANGE", 7: "PIC_ERR_ALIGNMENT",
    8: "PIC_ERR_CUDA", 9: "PIC_ERR_DEVICE_CHECK", 10: "PIC_ERR_UNSUPPORTED", 11: "PIC_ERR_BUSY",
}
PIC_KIND_GQA, PIC_KIND_MLA = 0, 1
PIC_PAIRING_NEOX_HALF, PIC_PAIRING_INTERLEAVED = 0, 1
PIC_SCALING_NONE, PIC_SCALING_LLAMA3 = 0, 1
PIC_KEY_BYTES = 32
PIC_DEV_BAD_BLOCK = 0x1
PIC_DEV_TIMEOUT = 0x2
PIC_DEV_BAD_TOKEN = 0x4
PIC_DEV_BAD_DOCS = 0x8
PIC_DEV_CAPACITY = 0x10
PIC_DEV_BAD_SPAN = 0x20
PIC_VARIANT_REGISTERS, PIC_VARIANT_BULK_PIPELINE = 0, 1
PIC_VARIANT_TENSOR_CORE_TMEM, PIC_VARIANT_WARP_MMA = 2, 3
PIC_SEG_COPY_POOL, PIC_SEG_COPY_BLOCKS, PIC_SEG_MAPPED = 0, 1, 2
PIC_ATTEND_FUSED, PIC_ATTEND_CACHE = 0, 1


class PicError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = STATUS_NAMES.get(status, f"PIC_ERR_{status}")
        super().__init__(f"{self.status_name}: {message}")


class pic_model_desc(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32), ("num_layers", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("rope_dim", ctypes.c_int32), ("rope_offset", ctypes.c_int32),
        ("pairing", ctypes.c_int32), ("block_size", ctypes.c_int32), ("scaling", ctypes.c_int32),
        ("llama3_orig_max_pos", ctypes.c_int32), ("rope_theta", ctypes.c_double),
        ("llama3_factor", ctypes.c_double), ("llama3_low_freq_factor", ctypes.c_double),
        ("llama3_high_freq_factor", ctypes.c_double), ("inv_freq", ctypes.POINTER(ctypes.c_double)),
    ]


class pic_request_desc(ctypes.Structure):
    _fields_ = [
        ("chunk_ids", ctypes.POINTER(ctypes.c_int32)), ("take_tokens", ctypes.POINTER(ctypes.c_int32)),
        ("dst_pos", ctypes.POINTER(ctypes.c_int32)), ("n_chunks", ctypes.c_int32),
        ("start_pos", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
        ("k_nonleading", ctypes.c_int32), ("k_leading", ctypes.c_int32), ("alias", ctypes.c_int32),
    ]


class pic_shift_seg(ctypes.Structure):
    _fields_ = [("req", ctypes.c_int32), ("start_pos", ctypes.c_int32),
                ("num_tokens", ctypes.c_int32), ("delta", ctypes.c_int32)]


_c_void_p = ctypes.c_void_p
_i32, _i64, _u32, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t
_P = ctypes.POINTER

_SIGNATURES = {
    "pic_abi_version": (_i32, []),
    "pic_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pic_last_error": (ctypes.c_char_p, [_c_void_p]),
    "pic_create": (ctypes.c_int, [_P(pic_model_desc), _i32, _P(_c_void_p)]),
    "pic_destroy": (None, [_c_void_p]),
    "pic_register_chunk": (ctypes.c_int, [_c_void_p, ctypes.c_char_p, _i64, _i32, _i32, _P(_i32), _P(_i32)]),
    "pic_register_chunk_blocks": (ctypes.c_int, [_c_void_p, ctypes.c_char_p, _P(_i32), _i32, _i32, _P(_i32),
                                                 _P(_i32)]),
    "pic_lookup_chunk": (ctypes.c_int, [_c_void_p, ctypes.c_char_p, _P(_i32)]),
    "pic_chunk_info": (ctypes.c_int, [_c_void_p, _i32, _P(_i64), _P(_i32), _P(_i32)]),
    "pic_unregister_chunk": (ctypes.c_int, [_c_void_p, _i32]),
    "pic_build_block_table": (ctypes.c_int, [_c_void_p, _P(pic_request_desc), _P(_i32), _i32, _P(_c_void_p)]),
    "pic_free_request": (ctypes.c_int, [_c_void_p, _c_void_p]),
    "pic_plan_info": (ctypes.c_int, [_c_void_p, _P(_i32), _P(_i32), _P(_i32), _P(_i32)]),
    "pic_plan_segment": (ctypes.c_int, [_c_void_p, _i32, _P(_i32), _P(_i64), _P(_i32), _P(_i32), _P(_i32)]),
    "pic_plan_segment_mode": (_i32, [_c_void_p, _i32]),
    "pic_workspace_bytes": (_sz, [_c_void_p, _P(_c_void_p), _i32]),
    "pic_stitch": (ctypes.c_int, [_c_void_p, _P(_c_void_p), _i32, _c_void_p, _c_void_p, _i64,
                                  _c_void_p, _c_void_p, _i64, _c_void_p, _i32, _c_void_p, _c_void_p,
                                  _i64, _c_void_p, _sz, _c_void_p]),
    "pic_stitch_noalloc": (ctypes.c_int, [_c_void_p, _P(_c_void_p), _i32, _c_void_p, _c_void_p, _i64,
                                          _c_void_p, _c_void_p, _i64, _c_void_p, _i32, _c_void_p,
                                          _c_void_p, _i64, _c_void_p, _c_void_p]),
    "pic_pool_read_rows": (ctypes.c_int, [_c_void_p, _P(_c_void_p), _i32, _P(_c_void_p), _i32, _P(_i64), _P(_i64)]),
    "pic_stage_pool": (ctypes.c_int, [_c_void_p, _P(_c_void_p), _i32, _P(_c_void_p), _i32, _c_void_p, _c_void_p,
                                      _i64, _c_void_p, _c_void_p, _i64, _P(_i64), _c_void_p]),
    "pic_stitch_staged_workspace_bytes": (_sz, [_c_void_p, _P(_c_void_p), _i32, _i32]),
    "pic_stitch_staged": (ctypes.c_int, [_c_void_p, _P(_c_void_p), _i32, _i32, _c_void_p, _c_void_p, _i64, _c_void_p,
                                         _c_void_p, _i64, _c_void_p, _c_void_p, _i64, _c_void_p, _i32, _c_void_p,
                                         _c_void_p, _i64, _c_void_p, _sz, _P(_i64), _c_void_p]),
    "pic_rerotate_workspace_bytes": (_sz, [_c_void_p, _P(pic_shift_seg), _i32]),
    "pic_rerotate_inplace": (ctypes.c_int, [_c_void_p, _c_void_p, _i64, _c_void_p, _i32, _i32,
                                            _P(pic_shift_seg), _i32, _c_void_p, _sz, _c_void_p]),
    "pic_recompute_indices": (ctypes.c_int, [_P(_c_void_p), _i32, _P(_i32), _P(_i32), _i64, _P(_i64)]),
    "pic_query_device_status": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _P(_u32)]),
    "pic_kernel_variant": (_i32, [_c_void_p, _i32]),
    "pic_attend_workspace_bytes": (_sz, [_c_void_p, _P(_c_void_p), _i32, _i32, _i32]),
    "pic_attend_decode": (ctypes.c_int, [_c_void_p, _P(_c_void_p), _i32, _i32, _c_void_p, _i32, ctypes.c_float,
                                         ctypes.c_float, _c_void_p, _c_void_p, _i64, _c_void_p, _c_void_p, _i64,
                                         _i32, _i32, _c_void_p, _c_void_p, _c_void_p, _sz, _c_void_p]),
    "pic_rotation_cossin": (ctypes.c_int, [_c_void_p, _c_void_p, _i32, _c_void_p, _c_void_p, _sz, _c_void_p]),
    "pic_cdc_workspace_bytes": (_sz, [_i64]),
    "pic_cdc_chunk": (ctypes.c_int, [_c_void_p, _i64, _c_void_p, _i32, _c_void_p, _i32, ctypes.c_uint64, _i32,
                                     _i32, ctypes.c_uint64, _c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p, _sz,
                                     _c_void_p]),
    "pic_fingerprint_spans": (ctypes.c_int, [_c_void_p, _i64, _c_void_p, _c_void_p, _i64, ctypes.c_uint64,
                                             _c_void_p, _c_void_p, _c_void_p]),
    "pic_s1_windows": (ctypes.c_int, [_i64, _i64, _i32, _P(_i64), _P(_i64), _i64, _P(_i64)]),
    "pic_debug_stall_next_launch": (ctypes.c_int, [_c_void_p, _i32, _u32]),
}

_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = False):
    """Loads libpic.so (building it first only when asked); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and (not os.path.exists(_build.LIB_PATH) or _build.is_stale()):
        _build.build()
    if not os.path.exists(_build.LIB_PATH):
        raise ImportError(f"libpic is not built ({_build.LIB_PATH} missing): run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(_build.LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(st: int, ctx=None):
    if st != PIC_OK:
        msg = load().pic_last_error(ctx)
        raise PicError(st, msg.decode() if msg else "")


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _i32_array(seq):
    if seq is None:
        return None
    a = (ctypes.c_int32 * len(seq))(*[int(x) for x in seq])
    return a


def _plan_array(plans):
    arr = (ctypes.c_void_p * max(1, len(plans)))()
    for i, p in enumerate(plans):
        arr[i] = p.value if isinstance(p, ctypes.c_void_p) else p
    return arr


# ------------------------------------------------------------------ context

def pic_abi_version() -> int:
    return load().pic_abi_version()


def pic_create(kind, num_layers, num_kv_heads, head_dim, rope_dim, rope_offset, pairing,
               block_size, rope_theta, num_cache_blocks, llama3=None, inv_freq=None):
    """Returns an opaque context handle (ctypes.c_void_p)."""
    d = pic_model_desc()
    d.kind, d.num_layers, d.num_kv_heads, d.head_dim = kind, num_layers, num_kv_heads, head_dim
    d.rope_dim, d.rope_offset, d.pairing, d.block_size = rope_dim, rope_offset, pairing, block_size
    d.rope_theta = float(rope_theta)
    keep = None
    if llama3:
        d.scaling = PIC_SCALING_LLAMA3
        d.llama3_factor = llama3["factor"]
        d.llama3_low_freq_factor = llama3["low_freq_factor"]
        d.llama3_high_freq_factor = llama3["high_freq_factor"]
        d.llama3_orig_max_pos = int(llama3["orig_max_pos"])
    if inv_freq is not None:
        keep = (ctypes.c_double * len(inv_freq))(*[float(x) for x in inv_freq])
        d.inv_freq = ctypes.cast(keep, ctypes.POINTER(ctypes.c_double))
    out = ctypes.c_void_p()
    st = load().pic_create(ctypes.byref(d), int(num_cache_blocks), ctypes.byref(out))
    _check(st, None)
    return out


def pic_destroy(ctx):
    load().pic_destroy(ctx)


def pic_last_error(ctx=None) -> str:
    return load().pic_last_error(ctx).decode()


# ----------------------------------------------------------------- registry

def pic_register_chunk(ctx, key: bytes, pool_token_offset: int, num_tokens: int, base_pos: int = 0):
    """Returns (chunk_id, is_new)."""
    if len(key) != PIC_KEY_BYTES:
        raise ValueError("key must be 32 bytes")
    cid, new = ctypes.c_int32(), ctypes.c_int32()
    _check(load().pic_register_chunk(ctx, key, int(pool_token_offset), int(num_tokens), int(base_pos),
                                     ctypes.byref(cid), ctypes.byref(new)), ctx)
    return cid.value, bool(new.value)


def pic_register_chunk_blocks(ctx, key: bytes, blocks, num_tokens: int, base_pos: int = 0):
    """Registers a chunk whose KV sits in the given paged-cache blocks.
    Returns (chunk_id, is_new)."""
    if len(key) != PIC_KEY_BYTES:
        raise ValueError("key must be 32 bytes")
    arr = _i32_array(list(blocks))
    cid, new = ctypes.c_int32(), ctypes.c_int32()
    _check(load().pic_register_chunk_blocks(ctx, key, ctypes.cast(arr, _P(_i32)), int(num_tokens), int(base_pos),
                                            ctypes.byref(cid), ctypes.byref(new)), ctx)
    return cid.value, bool(new.value)


def pic_lookup_chunk(ctx, key: bytes) -> int:
    cid = ctypes.c_int32()
    _check(load().pic_lookup_chunk(ctx, key, ctypes.byref(cid)), ctx)
    return cid.value


def pic_chunk_info(ctx, chunk_id: int):
    off, n, b = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
    _check(load().pic_chunk_info(ctx, chunk_id, ctypes.byref(off), ctypes.byref(n), ctypes.byref(b)), ctx)
    return off.value, n.value, b.value


def pic_unregister_chunk(ctx, chunk_id: int):
    _check(load().pic_unregister_chunk(ctx, chunk_id), ctx)


# ---------------------------------------------------------------- planning

def pic_build_block_table(ctx, chunk_ids, max_blocks: int, take_tokens=None, dst_pos=None,
                          start_pos: int = 0, total_tokens: int = 0, k_nonleading: int = 0,
                          k_leading: int = 0, alias: bool = False):
    """Returns (plan handle, block table as numpy int32[max_blocks])."""
    rq = pic_request_desc()
    ids = _i32_array(list(chunk_ids))
    take = _i32_array(take_tokens)
    pos = _i32_array(dst_pos)
    rq.chunk_ids = ctypes.cast(ids, _P(_i32)) if ids is not None else None
    rq.take_tokens = ctypes.cast(take, _P(_i32)) if take is not None else None
    rq.dst_pos = ctypes.cast(pos, _P(_i32)) if pos is not None else None
    rq.n_chunks = len(chunk_ids)
    rq.start_pos, rq.total_tokens = int(start_pos), int(total_tokens)
    rq.k_nonleading, rq.k_leading = int(k_nonleading), int(k_leading)
    rq.alias = 1 if alias else 0
    bt = np.empty(max(0, int(max_blocks)), dtype=np.int32)
    plan = ctypes.c_void_p()
    _check(load().pic_build_block_table(ctx, ctypes.byref(rq),
                                        bt.ctypes.data_as(_P(_i32)) if bt.size else None,
                                        int(max_blocks), ctypes.byref(plan)), ctx)
    return plan, bt


def pic_free_request(ctx, plan):
    _check(load().pic_free_request(ctx, plan), ctx)


def pic_plan_info(plan):
    t, b, s, r = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(load().pic_plan_info(plan, ctypes.byref(t), ctypes.byref(b), ctypes.byref(s), ctypes.byref(r)))
    return {"total_tokens": t.value, "num_blocks": b.value, "num_segments": s.value, "num_recompute": r.value}


def pic_plan_segment(plan, j: int):
    c, src, n, p, d = ctypes.c_int32(), ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check(load().pic_plan_segment(plan, j, ctypes.byref(c), ctypes.byref(src), ctypes.byref(n),
                                   ctypes.byref(p), ctypes.byref(d)))
    return {"chunk_id": c.value, "src_tok": src.value, "num_tokens": n.value, "dst_pos": p.value,
            "delta": d.value}


def pic_plan_segment_mode(plan, j: int) -> int:
    """PIC_SEG_COPY_POOL, PIC_SEG_COPY_BLOCKS or PIC_SEG_MAPPED."""
    return int(load().pic_plan_segment_mode(plan, int(j)))


def pic_recompute_indices(plans):
    """Host recompute list of a batch: (indptr int32[n+1], idx int32[count])."""
    arr = _plan_array(plans)
    count = ctypes.c_int64()
    _check(load().pic_recompute_indices(arr, len(plans), None, None, 0, ctypes.byref(count)))
    idx = np.empty(max(1, count.value), dtype=np.int32)
    indptr = np.empty(len(plans) + 1, dtype=np.int32)
    _check(load().pic_recompute_indices(arr, len(plans), idx.ctypes.data_as(_P(_i32)),
                                        indptr.ctypes.data_as(_P(_i32)), count.value, ctypes.byref(count)))
    return indptr, idx[:count.value]


# ------------------------------------------------------------------ stitch

def pic_workspace_bytes(ctx, plans) -> int:
    return int(load().pic_workspace_bytes(ctx, _plan_array(plans), len(plans)))


def _layer_stride_bytes(t):
    return t.stride(0) * t.element_size() if t is not None else 0


def pic_stitch(ctx, plans, k_pool, v_pool, k_cache, v_cache, block_tables, recompute_idx=None,
               recompute_indptr=None, workspace=None, stream=None):
    """Enqueues the stitch.  Tensors: pools [L][tokens][...], caches
    [L][blocks][block_size][...] (bf16, contiguous rows), block_tables int32
    [n_req][max_blocks] on the device, recompute outputs int32 or None,
    workspace uint8 with >= pic_workspace_bytes bytes."""
    arr = _plan_array(plans)
    _check_device_int32(block_tables, "block_tables")
    if block_tables.dim() != 2 or (len(plans) > 0 and block_tables.shape[0] < len(plans)):
        raise ValueError("block_tables must be [n_req][max_blocks] with a row per plan")
    if recompute_indptr is not None:
        _check_device_int32(recompute_indptr, "recompute_indptr")
        _check_device_int32(recompute_idx, "recompute_idx")
        if recompute_indptr.numel() < len(plans) + 1:
            raise ValueError("recompute_indptr needs n_req + 1 entries")
    for name, t in (("k_pool", k_pool), ("v_pool", v_pool), ("k_cache", k_cache), ("v_cache", v_cache)):
        _check_kv_buffer(t, name)
    pool_ls = _layer_stride_bytes(k_pool)
    cache_ls = _layer_stride_bytes(k_cache)
    if v_pool is not None and _layer_stride_bytes(v_pool) != pool_ls:
        raise ValueError("k_pool and v_pool must share a layer stride")
    if v_cache is not None and _layer_stride_bytes(v_cache) != cache_ls:
        raise ValueError("k_cache and v_cache must share a layer stride")
    cap = recompute_idx.numel() if recompute_idx is not None else 0
    st = load().pic_stitch(ctx, arr, len(plans), _ptr(k_pool), _ptr(v_pool), pool_ls,
                           _ptr(k_cache), _ptr(v_cache), cache_ls, _ptr(block_tables),
                           int(block_tables.shape[1]) if block_tables.dim() == 2 else int(block_tables.numel()),
                           _ptr(recompute_idx), _ptr(recompute_indptr), cap, _ptr(workspace),
                           workspace.numel() * workspace.element_size() if workspace is not None else 0,
                           _stream_handle(stream))
    _check(st, ctx)


def pic_pool_read_rows(ctx, plans, staged_plans=()):
    """(distinct pool rows outside those staged_plans read, pool rows read)
    of a batch, per layer."""
    d, r = ctypes.c_int64(), ctypes.c_int64()
    staged_plans = list(staged_plans)
    _check(load().pic_pool_read_rows(ctx, _plan_array(plans), len(plans),
                                     _plan_array(staged_plans) if staged_plans else None, len(staged_plans),
                                     ctypes.byref(d), ctypes.byref(r)), ctx)
    return d.value, r.value


def pic_stage_pool(ctx, plans, host_k_pool, host_v_pool, dev_k_pool, dev_v_pool, staged_plans=(),
                   stream=None) -> int:
    """Enqueues the copies of the pool rows the plans read, each once, from
    pinned host pools [L][tokens][...] into device pools of the same shape
    (v None for MLA), skipping the rows staged_plans read (staged by an
    earlier call).  Returns the bytes enqueued."""
    for name, t in (("host_k_pool", host_k_pool), ("host_v_pool", host_v_pool), ("dev_k_pool", dev_k_pool),
                    ("dev_v_pool", dev_v_pool)):
        _check_kv_buffer(t, name)
    hls, dls = _layer_stride_bytes(host_k_pool), _layer_stride_bytes(dev_k_pool)
    if host_v_pool is not None and _layer_stride_bytes(host_v_pool) != hls:
        raise ValueError("host_k_pool and host_v_pool must share a layer stride")
    if dev_v_pool is not None and _layer_stride_bytes(dev_v_pool) != dls:
        raise ValueError("dev_k_pool and dev_v_pool must share a layer stride")
    n = ctypes.c_int64()
    staged_plans = list(staged_plans)
    st = load().pic_stage_pool(ctx, _plan_array(plans), len(plans), _plan_array(staged_plans) if staged_plans else None,
                               len(staged_plans), _ptr(host_k_pool), _ptr(host_v_pool), hls,
                               _ptr(dev_k_pool), _ptr(dev_v_pool), dls, ctypes.byref(n), _stream_handle(stream))
    _check(st, ctx)
    return n.value


def pic_stitch_staged_workspace_bytes(ctx, plans, n_groups: int) -> int:
    return int(load().pic_stitch_staged_workspace_bytes(ctx, _plan_array(plans), len(plans), int(n_groups)))


def pic_stitch_staged(ctx, plans, host_k_pool, host_v_pool, dev_k_pool, dev_v_pool, k_cache, v_cache, block_tables,
                      recompute_idx=None, recompute_indptr=None, workspace=None, n_groups: int = 8,
                      stream=None) -> int:
    """pic_stage_pool + pic_stitch in one call, pipelined over n_groups
    groups of requests.  Pools as pic_stage_pool, the rest as pic_stitch;
    workspace >= pic_stitch_staged_workspace_bytes.  Returns the bytes
    staged."""
    arr = _plan_array(plans)
    _check_device_int32(block_tables, "block_tables")
    if block_tables.dim() != 2 or (len(plans) > 0 and block_tables.shape[0] < len(plans)):
        raise ValueError("block_tables must be [n_req][max_blocks] with a row per plan")
    if recompute_indptr is not None:
        _check_device_int32(recompute_indptr, "recompute_indptr")
        _check_device_int32(recompute_idx, "recompute_idx")
        if recompute_indptr.numel() < len(plans) + 1:
            raise ValueError("recompute_indptr needs n_req + 1 entries")
    for name, t in (("host_k_pool", host_k_pool), ("host_v_pool", host_v_pool), ("dev_k_pool", dev_k_pool),
                    ("dev_v_pool", dev_v_pool), ("k_cache", k_cache), ("v_cache", v_cache)):
        _check_kv_buffer(t, name)
    hls, dls, cls = _layer_stride_bytes(host_k_pool), _layer_stride_bytes(dev_k_pool), _layer_stride_bytes(k_cache)
    for a, b, what in ((host_v_pool, hls, "host pools"), (dev_v_pool, dls, "device pools"), (v_cache, cls, "caches")):
        if a is not None and _layer_stride_bytes(a) != b:
            raise ValueError(f"the K and V {what} must share a layer stride")
    cap = recompute_idx.numel() if recompute_idx is not None else 0
    n = ctypes.c_int64()
    st = load().pic_stitch_staged(ctx, arr, len(plans), int(n_groups), _ptr(host_k_pool), _ptr(host_v_pool), hls,
                                  _ptr(dev_k_pool), _ptr(dev_v_pool), dls, _ptr(k_cache), _ptr(v_cache), cls,
                                  _ptr(block_tables), int(block_tables.shape[1]), _ptr(recompute_idx),
                                  _ptr(recompute_indptr), cap, _ptr(workspace),
                                  workspace.numel() * workspace.element_size() if workspace is not None else 0,
                                  ctypes.byref(n), _stream_handle(stream))
    _check(st, ctx)
    return n.value


def pic_stitch_noalloc(ctx, plans, k_pool, v_pool, k_cache, v_cache, block_tables, recompute_idx=None,
                       recompute_indptr=None, status=None, stream=None):
    """pic_stitch for callers that cannot allocate device memory: same
    arguments minus the workspace (the library's own fixed 4 MiB device
    scratch is used; see include/pic.h).  ``status``: optional CUDA uint32
    tensor that receives this launch's device status word."""
    arr = _plan_array(plans)
    _check_device_int32(block_tables, "block_tables")
    if block_tables.dim() != 2 or (len(plans) > 0 and block_tables.shape[0] < len(plans)):
        raise ValueError("block_tables must be [n_req][max_blocks] with a row per plan")
    if recompute_indptr is not None:
        _check_device_int32(recompute_indptr, "recompute_indptr")
        _check_device_int32(recompute_idx, "recompute_idx")
        if recompute_indptr.numel() < len(plans) + 1:
            raise ValueError("recompute_indptr needs n_req + 1 entries")
    for name, t in (("k_pool", k_pool), ("v_pool", v_pool), ("k_cache", k_cache), ("v_cache", v_cache)):
        _check_kv_buffer(t, name)
    if status is not None and (not status.is_cuda or status.element_size() != 4 or status.numel() < 1):
        raise ValueError("status must be a CUDA tensor of at least one 32-bit element")
    pool_ls = _layer_stride_bytes(k_pool)
    cache_ls = _layer_stride_bytes(k_cache)
    if v_pool is not None and _layer_stride_bytes(v_pool) != pool_ls:
        raise ValueError("k_pool and v_pool must share a layer stride")
    if v_cache is not None and _layer_stride_bytes(v_cache) != cache_ls:
        raise ValueError("k_cache and v_cache must share a layer stride")
    cap = recompute_idx.numel() if recompute_idx is not None else 0
    st = load().pic_stitch_noalloc(ctx, arr, len(plans), _ptr(k_pool), _ptr(v_pool), pool_ls,
                                   _ptr(k_cache), _ptr(v_cache), cache_ls, _ptr(block_tables),
                                   int(block_tables.shape[1]), _ptr(recompute_idx), _ptr(recompute_indptr),
                                   cap, _ptr(status), _stream_handle(stream))
    _check(st, ctx)


def _check_device_int32(t, name):
    import torch
    if t is None or not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA int32 tensor")


def _rows_contiguous(t):
    """Everything but the layer axis is dense (the layer stride is passed separately)."""
    return t[0].is_contiguous() if t.dim() > 1 else t.is_contiguous()


def _check_kv_buffer(t, name):
    """Pools and caches: bf16 with contiguous rows, on the GPU or in pinned host memory."""
    if t is None:
        return
    if not _is_bf16(t) or not _rows_contiguous(t):
        raise ValueError(f"{name} must be a bf16 tensor with contiguous rows")
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name} must be a CUDA tensor or a pinned host tensor")


def _is_bf16(t):
    import torch
    return t.dtype == torch.bfloat16


def _shift_array(segs):
    arr = (pic_shift_seg * max(1, len(segs)))()
    for i, (req, start, n, delta) in enumerate(segs):
        arr[i].req, arr[i].start_pos, arr[i].num_tokens, arr[i].delta = int(req), int(start), int(n), int(delta)
    return arr


def pic_rerotate_workspace_bytes(ctx, segs) -> int:
    return int(load().pic_rerotate_workspace_bytes(ctx, _shift_array(segs), len(segs)))


def pic_rerotate_inplace(ctx, k_cache, block_tables, segs, workspace, stream=None):
    """segs: iterable of (req, start_pos, num_tokens, delta) on the host."""
    segs = list(segs)
    arr = _shift_array(segs)
    _check_device_int32(block_tables, "block_tables")
    _check_kv_buffer(k_cache, "k_cache")
    n_tables = int(block_tables.shape[0]) if block_tables.dim() == 2 else 1
    max_blocks = int(block_tables.shape[-1])
    st = load().pic_rerotate_inplace(ctx, _ptr(k_cache), _layer_stride_bytes(k_cache), _ptr(block_tables),
                                     n_tables, max_blocks, arr, len(segs), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, ctx)


def pic_query_device_status(ctx, workspace, stream=None, raise_on_device_error: bool = True) -> int:
    """Synchronizes the stream; returns the device status word (raises on a
    non-zero word with PIC_ERR_DEVICE_CHECK unless raise_on_device_error is
    False).  ctx may be None for a chunking workspace."""
    out = ctypes.c_uint32()
    st = load().pic_query_device_status(ctx, _ptr(workspace), _stream_handle(stream), ctypes.byref(out))
    if st == 9 and not raise_on_device_error:   # PIC_ERR_DEVICE_CHECK
        return out.value
    if st != PIC_OK:
        raise PicError(st, load().pic_last_error(ctx).decode())
    return out.value


# ------------------------------------------------- content-defined chunking

def pic_cdc_workspace_bytes(n_tokens: int) -> int:
    return int(load().pic_cdc_workspace_bytes(int(n_tokens)))


def _check_device(t, dtype, name, allow_none=False):
    import torch
    if t is None:
        if allow_none:
            return
        raise ValueError(f"{name} is required")
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def pic_cdc_chunk(tokens, doc_offsets, gear, threshold: int, chunk_indptr, chunk_ends, fingerprints=None,
                  min_len: int = 0, max_len: int = 0, seed: int = 0, workspace=None, stream=None):
    """Content-defined chunking of the documents [offsets[d], offsets[d + 1]) of
    ``tokens`` (CUDA int32); ``doc_offsets`` CUDA int64 [n_docs + 1]; ``gear``
    CUDA uint64 (or int64 holding the same bits) [vocab].  Writes
    ``chunk_indptr`` (int64 [n_docs + 1]), ``chunk_ends`` (int64 [capacity])
    and ``fingerprints`` (int64/uint64 [capacity], optional).  The workspace
    is allocated here if not given.  Returns the workspace (its status word is
    read with pic_query_device_status(None, workspace))."""
    import torch
    _check_device(tokens, torch.int32, "tokens")
    _check_device(doc_offsets, torch.int64, "doc_offsets")
    if gear.dtype not in (torch.int64, torch.uint64) or not gear.is_cuda or not gear.is_contiguous():
        raise ValueError("gear must be a contiguous CUDA 64-bit integer tensor")
    _check_device(chunk_indptr, torch.int64, "chunk_indptr")
    _check_device(chunk_ends, torch.int64, "chunk_ends")
    if fingerprints is not None and (fingerprints.dtype not in (torch.int64, torch.uint64) or not fingerprints.is_cuda
                                     or not fingerprints.is_contiguous()):
        raise ValueError("fingerprints must be a contiguous CUDA 64-bit integer tensor")
    n_docs = doc_offsets.numel() - 1
    if n_docs < 0 or chunk_indptr.numel() < n_docs + 1:
        raise ValueError("doc_offsets needs n_docs + 1 entries and chunk_indptr as many")
    cap = chunk_ends.numel()
    if fingerprints is not None and fingerprints.numel() < cap:
        raise ValueError("fingerprints must hold as many entries as chunk_ends")
    if workspace is None:
        workspace = torch.empty(max(1, pic_cdc_workspace_bytes(tokens.numel())), dtype=torch.uint8,
                                device=tokens.device)
    st = load().pic_cdc_chunk(_ptr(tokens), tokens.numel(), _ptr(doc_offsets), n_docs, _ptr(gear), gear.numel(),
                              int(threshold) & ((1 << 64) - 1), int(min_len), int(max_len),
                              int(seed) & ((1 << 64) - 1), _ptr(chunk_indptr), _ptr(chunk_ends),
                              _ptr(fingerprints), cap, _ptr(workspace), workspace.numel(), _stream_handle(stream))
    _check(st, None)
    return workspace


def pic_fingerprint_spans(tokens, starts, ends, out, status, seed: int = 0, stream=None):
    """XXH64 of token spans [starts[k], ends[k]) into ``out`` (CUDA 64-bit
    integers); ``status`` is a CUDA 32-bit tensor that receives PIC_DEV_BAD_SPAN."""
    import torch
    _check_device(tokens, torch.int32, "tokens")
    _check_device(starts, torch.int64, "starts")
    _check_device(ends, torch.int64, "ends")
    n = starts.numel()
    if ends.numel() != n or out.numel() < n or out.element_size() != 8 or not out.is_cuda:
        raise ValueError("starts, ends and out must hold one 64-bit entry per span")
    if not status.is_cuda or status.element_size() != 4:
        raise ValueError("status must be a CUDA 32-bit tensor")
    st = load().pic_fingerprint_spans(_ptr(tokens), tokens.numel(), _ptr(starts), _ptr(ends), n,
                                      int(seed) & ((1 << 64) - 1), _ptr(out), _ptr(status), _stream_handle(stream))
    _check(st, None)


def pic_s1_windows(begin: int, end: int, window: int = 128):
    """(starts, ends) of the fixed windows covering [begin, end), as lists."""
    lib_ = load()
    n = ctypes.c_int64()
    _check(lib_.pic_s1_windows(int(begin), int(end), int(window), None, None, 0, ctypes.byref(n)), None)
    a = (ctypes.c_int64 * max(1, n.value))()
    b = (ctypes.c_int64 * max(1, n.value))()
    _check(lib_.pic_s1_windows(int(begin), int(end), int(window), a, b, n.value, ctypes.byref(n)), None)
    return list(a[:n.value]), list(b[:n.value])


def pic_attend_workspace_bytes(ctx, plans, num_q_heads: int, num_layers: int) -> int:
    return int(load().pic_attend_workspace_bytes(ctx, _plan_array(plans), len(plans), int(num_q_heads),
                                                 int(num_layers)))


def pic_attend_decode(ctx, plans, source, q, softmax_scale, k_pool, v_pool, k_cache, v_cache, out, lse=None,
                      workspace=None, sink_bias=0.0, layer_begin=0, stream=None):
    """One decode step of attention over each plan's context.  q: CUDA bf16
    [num_layers][n_req][num_q_heads][head_dim]; out: CUDA float32 of the same
    shape (MLA: [..][512], the latent); lse: CUDA float32
    [num_layers][n_req][num_q_heads] or None.  MLA: v_pool and v_cache are None."""
    num_layers, n_req, hq = int(q.shape[0]), int(q.shape[1]), int(q.shape[2])
    if n_req != len(plans):
        raise ValueError("q holds one row per plan")
    st = load().pic_attend_decode(ctx, _plan_array(plans), len(plans), int(source), _ptr(q), hq,
                                  float(softmax_scale), float(sink_bias), _ptr(k_pool), _ptr(v_pool),
                                  _layer_stride_bytes(k_pool), _ptr(k_cache), _ptr(v_cache),
                                  _layer_stride_bytes(k_cache), int(layer_begin), num_layers, _ptr(out), _ptr(lse),
                                  _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _stream_handle(stream))
    _check(st, ctx)


def pic_debug_stall_next_launch(ctx, stall_tile: int, max_spins: int = 0):
    """Test hook: the next bulk-pipeline stitch on ctx leaves tile stall_tile
    of its first CTA without copies, so its bounded waits run out and raise
    PIC_DEV_TIMEOUT (see include/pic.h)."""
    _check(load().pic_debug_stall_next_launch(ctx, int(stall_tile), int(max_spins)), ctx)


def pic_kernel_variant(ctx, mode: int) -> int:
    """Kernel a context launches.  Modes 0 (stitch) and 1 (in-place shift):
    PIC_VARIANT_REGISTERS or PIC_VARIANT_BULK_PIPELINE.  Mode 2 (decode
    attention): PIC_VARIANT_TENSOR_CORE_TMEM (MLA on tcgen05) or
    PIC_VARIANT_WARP_MMA."""
    return int(load().pic_kernel_variant(ctx, int(mode)))


def pic_rotation_cossin(ctx, deltas, out, workspace, stream=None):
    """deltas: int32 device tensor [n]; out: float32 device tensor [n][rope_dim/2][2]."""
    st = load().pic_rotation_cossin(ctx, _ptr(deltas), int(deltas.numel()), _ptr(out), _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(st, ctx)


# ----------------------------------------------------------- convenience

@dataclass
class ModelSpec:
    """Geometry + RoPE settings (mirrors pic_model_desc)."""
    kind: int
    num_layers: int
    num_kv_heads: int
    head_dim: int
    rope_dim: int
    rope_offset: int
    pairing: int
    block_size: int
    rope_theta: float
    llama3: dict | None = None
    inv_freq: list | None = None

    @property
    def row_bytes(self) -> int:
        return self.num_kv_heads * self.head_dim * 2


def model_spec_from(model) -> ModelSpec:
    """ModelSpec from any object with the workload-model attributes."""
    return ModelSpec(
        kind=PIC_KIND_GQA if model.kind == "gqa" else PIC_KIND_MLA,
        num_layers=model.num_layers, num_kv_heads=model.num_kv_heads, head_dim=model.head_dim,
        rope_dim=model.rope_dim, rope_offset=model.rope_offset,
        pairing=PIC_PAIRING_NEOX_HALF if model.pairing == "neox" else PIC_PAIRING_INTERLEAVED,
        block_size=model.block_size, rope_theta=model.rope_theta, llama3=model.llama3)


def create_from_spec(spec: ModelSpec, num_cache_blocks: int):
    return pic_create(spec.kind, spec.num_layers, spec.num_kv_heads, spec.head_dim, spec.rope_dim,
                      spec.rope_offset, spec.pairing, spec.block_size, spec.rope_theta,
                      num_cache_blocks, llama3=spec.llama3, inv_freq=spec.inv_freq)
