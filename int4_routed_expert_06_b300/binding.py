"""ctypes binding of libmoe_int4.so: the same entry points as include/moe_int4.h.

Argument marshalling only: tensors become raw pointers, streams become
``cudaStream_t`` handles (default: torch's current stream), non-OK statuses
raise :class:`MoEError`.  Every step of the layer runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback, and importing a function whose
library is missing raises immediately.

Helpers at the end (:func:`config_for`, :class:`DeviceLayer`) only lay
weights out in the library's fixed-stride blob format, using the offsets that
``moe_blob_layout_get`` returns.
"""
from __future__ import annotations

import ctypes as C
import os
import re
from typing import Dict, Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmoe_int4.so")
HEADER = os.path.join(os.path.dirname(_PKG), "include", "moe_int4.h")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_OOM = 0, 1, 2, 3, 4
MOE_ERR_TIMEOUT, MOE_ERR_POOL_EXHAUSTED, MOE_ERR_NOT_RESIDENT, MOE_ERR_DEVICE_FAULT = 5, 6, 7, 8
MOE_F32, MOE_BF16, MOE_F16 = 0, 1, 2
_DTYPE = {"f32": MOE_F32, "bf16": MOE_BF16, "f16": MOE_F16}


class MoEError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"moe status {status}: {message}")
        self.status = status
        self.message = message


# ------------------------------------------------------------------ structs

class moe_config(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("hidden", "n_experts", "top_k", "inter", "shared_inter",
                                         "group_size", "act_dtype", "router_dtype", "qscale_dtype", "bits")]


class moe_qmat(C.Structure):
    _fields_ = [("q", C.c_void_p), ("scale", C.c_void_p), ("bias", C.c_void_p)]


class moe_expert(C.Structure):
    _fields_ = [("gate", moe_qmat), ("up", moe_qmat), ("down", moe_qmat)]


class moe_blob_layout(C.Structure):
    _fields_ = [(n, C.c_size_t) for n in ("q_gate", "q_up", "q_down", "s_gate", "b_gate", "s_up",
                                          "b_up", "s_down", "b_down", "bytes")]


class moe_layer(C.Structure):
    _fields_ = [("w_router", C.c_void_p), ("router_bias", C.c_void_p), ("w_shared_gate", C.c_void_p),
                ("shared_blob", C.c_void_p), ("pool", C.c_void_p), ("expert_stride", C.c_size_t),
                ("slot_table", C.c_void_p), ("n_slots", C.c_int32)]


class moe_pool_stats(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("lookups", "hits", "misses", "evictions", "bytes_filled",
                                         "exposed_copy_ns")]


class moe_resident_weights(C.Structure):
    _fields_ = [("w_router", C.c_void_p), ("router_bias", C.c_void_p), ("w_shared_gate", C.c_void_p),
                ("shared_blob", C.c_void_p)]


# ------------------------------------------------------------------ loading

_lib = None
_P, _Z, _I, _CP = C.c_void_p, C.c_size_t, C.c_int32, C.POINTER

_SIGS = {
    "moe_blob_layout_get": (_I, [_CP(moe_config), _I, _CP(moe_blob_layout)]),
    "moe_pack_expert": (_I, [_CP(moe_config), _I, _CP(moe_expert), _P]),
    "moe_route_workspace_bytes": (_Z, [_CP(moe_config), _I]),
    "moe_bucket_workspace_bytes": (_Z, [_CP(moe_config), _I]),
    "moe_expert_workspace_bytes": (_Z, [_CP(moe_config), _I]),
    "moe_layer_workspace_bytes": (_Z, [_CP(moe_config), _I]),
    "moe_route": (_I, [_CP(moe_config), _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_bucket": (_I, [_CP(moe_config), _P, _I, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_expert_forward": (_I, [_CP(moe_config), _CP(moe_expert), _I, _P, _I, _P, _P, _P, _Z, _P]),
    "moe_experts_forward": (_I, [_CP(moe_config), _CP(moe_layer), _P, _I, _P, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_layer_forward": (_I, [_CP(moe_config), _CP(moe_layer), _P, _I, _P, _P, _P, _P, _P, _Z, _P]),
    "moe_layer_forward_noalloc": (_I, [_CP(moe_config), _CP(moe_layer), _P, _I, _P, _P, _P, _P, _P]),
    "slot_pool_create": (_I, [_CP(moe_config), _I, _I, _P, _Z, _P, _Z, _P, _CP(_P)]),
    "slot_pool_lookup": (_I, [_P, _I, _P, _I, _P, _P, _CP(_I)]),
    "slot_pool_fill": (_I, [_P, _I, _P, _I, _P]),
    "slot_pool_layer": (_I, [_P, _I, _CP(_P), _CP(_P)]),
    "slot_pool_table_host": (_I, [_P, _I, _P]),
    "slot_pool_stats": (_I, [_P, _CP(moe_pool_stats)]),
    "moe_pooled_layer_forward": (_I, [_CP(moe_config), _P, _I, _CP(moe_resident_weights), _P, _I, _P, _P, _P,
                                      _P, _Z, _P]),
    "slot_pool_destroy": (None, [_P]),
    "slot_pool_set_policy": (_I, [_P, _I]),
    "slot_pool_enable_device": (_I, [_P]),
    "slot_pool_create_file": (_I, [_CP(moe_config), _I, _I, _P, _Z, C.c_char_p, _Z, _Z, _I, _P, _CP(_P)]),
    "slot_pool_file_stats": (_I, [_P, _CP(C.c_int64), _CP(C.c_int64), _CP(_I)]),
    "slot_pool_step_device": (_I, [_P, _I, _P, _I, _P]),
    "moe_get_device_error": (_I, [_P]),
    "moe_last_error_message": (C.c_char_p, []),
    "moe_version": (C.c_char_p, []),
    "moe_set_kernel_path": (_I, [_I]),
    "moe_debug_set_waits": (_I, [C.c_uint64, _I]),
}


def lib() -> C.CDLL:
    """Load libmoe_int4.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing; build it with "
                              "`python -m int4_routed_expert_06_b300.build`")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def header_functions() -> list:
    """Names of every function the public header declares."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w ]*?\**\s*\**\b(moe_\w+|slot_pool_\w+)\s*\(",
                                 txt, flags=re.M)))


def _check(st: int, what: str):
    if st != MOE_OK:
        msg = lib().moe_last_error_message().decode(errors="replace")
        raise MoEError(st, msg if msg.startswith(what) else f"{what}: {msg}")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, torch.Tensor):
        if not t.is_contiguous():
            # the C ABI takes dense row-major arrays; a strided view would be
            # read as if it were dense
            raise ValueError(f"tensor of shape {tuple(t.shape)} and strides {t.stride()} is not contiguous")
        return t.data_ptr()
    raise TypeError(f"cannot pass {type(t)} as a pointer")


def _stream(s) -> Optional[int]:
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, torch.cuda.Stream):
        return s.cuda_stream
    return int(s)


# ------------------------------------------------------------------ entry points

def moe_blob_layout_get(cfg: moe_config, inter: int) -> moe_blob_layout:
    out = moe_blob_layout()
    _check(lib().moe_blob_layout_get(C.byref(cfg), inter, C.byref(out)), "moe_blob_layout_get")
    return out


def moe_pack_expert(cfg: moe_config, inter: int, expert: moe_expert, dst_host) -> None:
    _check(lib().moe_pack_expert(C.byref(cfg), inter, C.byref(expert), _ptr(dst_host)), "moe_pack_expert")


def moe_route_workspace_bytes(cfg, T):
    return lib().moe_route_workspace_bytes(C.byref(cfg), T)


def moe_bucket_workspace_bytes(cfg, T):
    return lib().moe_bucket_workspace_bytes(C.byref(cfg), T)


def moe_expert_workspace_bytes(cfg, T):
    return lib().moe_expert_workspace_bytes(C.byref(cfg), T)


def moe_layer_workspace_bytes(cfg, T):
    return lib().moe_layer_workspace_bytes(C.byref(cfg), T)


def moe_route(cfg, x, T, w_router, router_bias, w_shared_gate, topk_idx, topk_w, shared_gate_logit,
              logits_out=None, workspace=None, ws_bytes=0, stream=None):
    _check(lib().moe_route(C.byref(cfg), _ptr(x), T, _ptr(w_router), _ptr(router_bias), _ptr(w_shared_gate),
                           _ptr(topk_idx), _ptr(topk_w), _ptr(shared_gate_logit), _ptr(logits_out),
                           _ptr(workspace), ws_bytes, _stream(stream)), "moe_route")


def moe_bucket(cfg, topk_idx, T, counts, offsets, perm_tok, perm_rank, workspace, ws_bytes, stream=None):
    _check(lib().moe_bucket(C.byref(cfg), _ptr(topk_idx), T, _ptr(counts), _ptr(offsets), _ptr(perm_tok),
                            _ptr(perm_rank), _ptr(workspace), ws_bytes, _stream(stream)), "moe_bucket")


def moe_expert_forward(cfg, expert: moe_expert, inter, x, T, y, y_f32, workspace, ws_bytes, stream=None):
    _check(lib().moe_expert_forward(C.byref(cfg), C.byref(expert), inter, _ptr(x), T, _ptr(y), _ptr(y_f32),
                                    _ptr(workspace), ws_bytes, _stream(stream)), "moe_expert_forward")


def moe_experts_forward(cfg, layer: moe_layer, x, T, topk_idx, topk_w, shared_gate_logit, y, y_f32,
                        workspace, ws_bytes, stream=None):
    _check(lib().moe_experts_forward(C.byref(cfg), C.byref(layer), _ptr(x), T, _ptr(topk_idx), _ptr(topk_w),
                                     _ptr(shared_gate_logit), _ptr(y), _ptr(y_f32), _ptr(workspace), ws_bytes,
                                     _stream(stream)), "moe_experts_forward")


def moe_layer_forward(cfg, layer: moe_layer, x, T, y, y_f32=None, topk_idx_out=None, topk_w_out=None,
                      workspace=None, ws_bytes=0, stream=None):
    _check(lib().moe_layer_forward(C.byref(cfg), C.byref(layer), _ptr(x), T, _ptr(y), _ptr(y_f32),
                                   _ptr(topk_idx_out), _ptr(topk_w_out), _ptr(workspace), ws_bytes,
                                   _stream(stream)), "moe_layer_forward")


def moe_layer_forward_noalloc(cfg, layer: moe_layer, x, T, y, y_f32=None, topk_idx_out=None, topk_w_out=None,
                              stream=None):
    """moe_layer_forward with the library's built-in scratch (no workspace argument)."""
    _check(lib().moe_layer_forward_noalloc(C.byref(cfg), C.byref(layer), _ptr(x), T, _ptr(y), _ptr(y_f32),
                                           _ptr(topk_idx_out), _ptr(topk_w_out), _stream(stream)),
           "moe_layer_forward_noalloc")


def slot_pool_create(cfg, n_layers, slots_per_layer, pool_dev, pool_bytes, backing_host, expert_stride,
                     side_stream=None) -> int:
    out = C.c_void_p()
    _check(lib().slot_pool_create(C.byref(cfg), n_layers, slots_per_layer, _ptr(pool_dev), pool_bytes,
                                  _ptr(backing_host), expert_stride,
                                  _stream(side_stream) if side_stream is not None else None, C.byref(out)),
           "slot_pool_create")
    return out.value


def slot_pool_lookup(pool: int, layer: int, expert_ids):
    """-> (slots list, miss ids list).  expert_ids: a sequence of ints (host)."""
    n = len(expert_ids)
    ids = (C.c_int32 * max(n, 1))(*expert_ids)
    slots = (C.c_int32 * max(n, 1))()
    miss = (C.c_int32 * max(n, 1))()
    n_miss = C.c_int32(0)
    _check(lib().slot_pool_lookup(pool, layer, ids, n, slots, miss, C.byref(n_miss)), "slot_pool_lookup")
    return list(slots)[:n], list(miss)[: n_miss.value]


def slot_pool_fill(pool: int, layer: int, miss_ids, done_event=None):
    n = len(miss_ids)
    ids = (C.c_int32 * max(n, 1))(*miss_ids)
    ev = None if done_event is None else done_event.cuda_event
    _check(lib().slot_pool_fill(pool, layer, ids, n, ev), "slot_pool_fill")


def slot_pool_layer(pool: int, layer: int):
    t, b = C.c_void_p(), C.c_void_p()
    _check(lib().slot_pool_layer(pool, layer, C.byref(t), C.byref(b)), "slot_pool_layer")
    return t.value, b.value


def slot_pool_table_host(pool: int, layer: int, n_experts: int):
    out = (C.c_int32 * n_experts)()
    _check(lib().slot_pool_table_host(pool, layer, out), "slot_pool_table_host")
    return list(out)


def slot_pool_stats(pool: int) -> dict:
    s = moe_pool_stats()
    _check(lib().slot_pool_stats(pool, C.byref(s)), "slot_pool_stats")
    return {n: getattr(s, n) for n, _ in moe_pool_stats._fields_}


def moe_pooled_layer_forward(cfg, pool: int, layer: int, weights: moe_resident_weights, x, T, y, y_f32,
                             topk_idx_out, workspace, ws_bytes, stream=None):
    _check(lib().moe_pooled_layer_forward(C.byref(cfg), pool, layer, C.byref(weights), _ptr(x), T, _ptr(y),
                                          _ptr(y_f32), _ptr(topk_idx_out), _ptr(workspace), ws_bytes,
                                          _stream(stream)), "moe_pooled_layer_forward")


MOE_POOL_LFU_RECENCY, MOE_POOL_LRU, MOE_POOL_LFU = 0, 1, 2


def slot_pool_set_policy(pool: int, policy: int) -> None:
    _check(lib().slot_pool_set_policy(pool, policy), "slot_pool_set_policy")


def slot_pool_create_file(cfg, n_layers, slots_per_layer, pool_dev, pool_bytes, path: str, file_offset: int,
                          file_stride: int, readers: int = 4, side_stream=None) -> int:
    out = C.c_void_p()
    _check(lib().slot_pool_create_file(C.byref(cfg), n_layers, slots_per_layer, _ptr(pool_dev), pool_bytes,
                                       path.encode(), file_offset, file_stride, readers,
                                       _stream(side_stream) if side_stream is not None else None, C.byref(out)),
           "slot_pool_create_file")
    return out.value


def slot_pool_file_stats(pool: int) -> dict:
    b, ns, d = C.c_int64(0), C.c_int64(0), C.c_int32(0)
    _check(lib().slot_pool_file_stats(pool, C.byref(b), C.byref(ns), C.byref(d)), "slot_pool_file_stats")
    return {"bytes_read": b.value, "read_ns": ns.value, "direct": bool(d.value)}


def slot_pool_enable_device(pool: int) -> None:
    _check(lib().slot_pool_enable_device(pool), "slot_pool_enable_device")


def slot_pool_step_device(pool: int, layer: int, ids_dev, n: int, stream=None) -> None:
    _check(lib().slot_pool_step_device(pool, layer, _ptr(ids_dev), n, _stream(stream)), "slot_pool_step_device")


def slot_pool_destroy(pool: int) -> None:
    lib().slot_pool_destroy(pool)


def moe_get_device_error(stream=None) -> int:
    """Status code of the device error word (read and cleared); 0 = none."""
    return lib().moe_get_device_error(_stream(stream))


def moe_last_error_message() -> str:
    return lib().moe_last_error_message().decode(errors="replace")


def moe_version() -> str:
    return lib().moe_version().decode()


def moe_set_kernel_path(path: int) -> None:
    _check(lib().moe_set_kernel_path(path), "moe_set_kernel_path")


def moe_debug_set_waits(wait_ns: int, extra_arrivals: int) -> None:
    _check(lib().moe_debug_set_waits(wait_ns, extra_arrivals), "moe_debug_set_waits")


# ------------------------------------------------------------------ marshalling helpers

def config_for(shape) -> moe_config:
    """moe_config of a synth.MoEShape."""
    return moe_config(shape.hidden, shape.n_experts, shape.top_k, shape.inter, shape.shared_inter, shape.group,
                      _DTYPE[shape.act], _DTYPE[shape.router], _DTYPE[shape.qscale], getattr(shape, "bits", 4))


_ARRAYS = ("q_gate", "q_up", "q_down", "s_gate", "b_gate", "s_up", "b_up", "s_down", "b_down")


def pack_blobs(cfg: moe_config, inter: int, mats: Dict[str, torch.Tensor], slots: torch.Tensor,
               n_slots: int, stride: int, prefix: str = "", out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Lay experts out as fixed-stride blobs: expert e goes to slot slots[e]
    of a [n_slots, stride] uint8 buffer on the arrays' device."""
    lay = moe_blob_layout_get(cfg, inter)
    dev = mats[prefix + "q_gate"].device
    if out is None:
        out = torch.zeros((n_slots, stride), dtype=torch.uint8, device=dev)
    sl = slots.to(device=dev, dtype=torch.long)
    for name in _ARRAYS:
        a = mats[prefix + name]
        n = a.shape[0]
        flat = a.contiguous().view(n, -1).view(torch.uint8)
        off = getattr(lay, name)
        out[sl, off:off + flat.shape[1]] = flat
    return out


def expert_struct(mats: Dict[str, torch.Tensor], e: int, prefix: str = "") -> moe_expert:
    """moe_expert of expert e of a stacked MLX-form dict (pointers into the tensors)."""
    def qm(m):
        return moe_qmat(mats[prefix + "q_" + m][e].data_ptr(), mats[prefix + "s_" + m][e].data_ptr(),
                        mats[prefix + "b_" + m][e].data_ptr())
    return moe_expert(qm("gate"), qm("up"), qm("down"))


class DeviceLayer:
    """A layer resident in one HBM pool of fixed-stride expert blobs.

    layer: synth.make_layer output (any device); slots: [E] int32 expert ->
    slot table (every expert resident); replicas: independent copies of the
    whole layer (pool, shared blob, router) at different addresses, so that a
    decode loop can rotate through them and not be served from L2.
    """

    def __init__(self, shape, layer: dict, slots: torch.Tensor, device="cuda", replicas: int = 1):
        self.shape, self.cfg = shape, config_for(shape)
        lay = moe_blob_layout_get(self.cfg, shape.inter)
        self.stride = (lay.bytes + 255) // 256 * 256
        self.n_slots = int(slots.max()) + 1
        dev_layer = {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in layer.items()}
        base = pack_blobs(self.cfg, shape.inter, dev_layer, slots, self.n_slots, self.stride)
        self.shared_stride = 0
        sh = None
        if shape.shared_inter > 0:
            lsh = moe_blob_layout_get(self.cfg, shape.shared_inter)
            self.shared_stride = (lsh.bytes + 255) // 256 * 256
            sh = pack_blobs(self.cfg, shape.shared_inter, dev_layer, torch.zeros(1, dtype=torch.int32), 1,
                            self.shared_stride, prefix="shared_")
        self.replicas = []
        for r in range(replicas):
            rep = {
                "pool": base if r == 0 else base.clone(),
                "shared": None if sh is None else (sh if r == 0 else sh.clone()),
                "w_router": dev_layer["w_router"].contiguous() if r == 0 else dev_layer["w_router"].clone(),
                "w_shared_gate": dev_layer["w_shared_gate"].contiguous() if r == 0
                else dev_layer["w_shared_gate"].clone(),
                "router_bias": None if dev_layer.get("router_bias") is None else dev_layer["router_bias"].clone(),
                "slots": slots.to(device=device, dtype=torch.int32).clone(),
            }
            rep["struct"] = self._struct(rep)
            self.replicas.append(rep)

    def _struct(self, rep) -> moe_layer:
        has_sh = self.shape.shared_inter > 0
        return moe_layer(rep["w_router"].data_ptr(),
                         rep["router_bias"].data_ptr() if rep["router_bias"] is not None else None,
                         rep["w_shared_gate"].data_ptr() if has_sh else None,
                         rep["shared"].data_ptr() if has_sh else None,
                         rep["pool"].data_ptr(), self.stride, rep["slots"].data_ptr(), self.n_slots)

    def struct(self, r: int = 0) -> moe_layer:
        return self.replicas[r]["struct"]
