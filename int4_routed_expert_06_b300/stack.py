"""A stack of MoE layers served from a bounded HBM expert pool.

Memory plumbing around the C-ABI: a pinned host backing store holding every
layer's expert blobs at a fixed stride, the device pool buffer, the resident
part of each layer (router, shared gate, shared expert) and the side stream
fills run on.  Each layer step is one ``moe_pooled_layer_forward`` call; the
routing, the LFU+recency policy, the fills and the expert kernels all run in
the library, the policy on the host, or (device_policy=True) as kernels on
the caller's stream, with the fills read from the pinned backing store.
"""
from __future__ import annotations

import os
from typing import Callable, Dict, List, Optional

import torch

from . import binding as B


class PooledStack:
    def __init__(self, shape, n_layers: int, slots_per_layer: int,
                 layer_weights: Callable[[int], Dict[str, torch.Tensor]], device: str = "cuda",
                 device_policy: bool = False, file_path: Optional[str] = None, readers: int = 4):
        self.shape, self.cfg = shape, B.config_for(shape)
        self.L, self.S, self.E = n_layers, slots_per_layer, shape.n_experts
        lay = B.moe_blob_layout_get(self.cfg, shape.inter)
        self.blob_bytes = lay.bytes
        self.stride = (lay.bytes + 255) // 256 * 256
        # backing store: pinned host memory, or (file_path) a file of 4 KiB-aligned records
        self.file_path = file_path
        self.file_stride = (lay.bytes + 4095) // 4096 * 4096
        self.backing = None if file_path else torch.empty((n_layers, self.E, self.stride), dtype=torch.uint8,
                                                           pin_memory=True)
        fh = open(file_path, "wb") if file_path else None
        self.pool = torch.empty((n_layers * slots_per_layer * self.stride,), dtype=torch.uint8, device=device)
        ident = torch.arange(self.E, dtype=torch.int32)
        self.resident: List[dict] = []
        for l in range(n_layers):
            w = layer_weights(l)
            if fh is not None:
                blobs = B.pack_blobs(self.cfg, shape.inter, w, ident, self.E, self.file_stride)
                fh.write(blobs.cpu().numpy().tobytes())
            else:
                blobs = B.pack_blobs(self.cfg, shape.inter, w, ident, self.E, self.stride)
                self.backing[l].copy_(blobs)
            del blobs
            sh_lay = B.moe_blob_layout_get(self.cfg, shape.shared_inter)
            sh_stride = (sh_lay.bytes + 255) // 256 * 256
            shared = B.pack_blobs(self.cfg, shape.shared_inter, w, torch.zeros(1, dtype=torch.int32), 1,
                                  sh_stride, prefix="shared_")
            r = {"w_router": w["w_router"].contiguous(), "w_shared_gate": w["w_shared_gate"].contiguous(),
                 "router_bias": w.get("router_bias"), "shared": shared}
            r["struct"] = B.moe_resident_weights(
                r["w_router"].data_ptr(), r["router_bias"].data_ptr() if r["router_bias"] is not None else None,
                r["w_shared_gate"].data_ptr(), shared.data_ptr())
            self.resident.append(r)
        self.side = torch.cuda.Stream()
        if fh is not None:
            fh.flush()
            os.fsync(fh.fileno())
            os.posix_fadvise(fh.fileno(), 0, 0, os.POSIX_FADV_DONTNEED)  # reads come from the device, not RAM
            fh.close()
            self.handle = B.slot_pool_create_file(self.cfg, n_layers, slots_per_layer, self.pool, self.pool.numel(),
                                                  file_path, 0, self.file_stride, readers, self.side)
        else:
            self.handle = B.slot_pool_create(self.cfg, n_layers, slots_per_layer, self.pool, self.pool.numel(),
                                             self.backing, self.stride, self.side)
        self.device_policy = device_policy
        if device_policy:  # lookup and fills as kernels on the caller's stream: no host round trip
            B.slot_pool_enable_device(self.handle)
        self.ws_bytes = 0
        self.ws = None

    def workspace(self, T: int) -> torch.Tensor:
        nb = B.moe_layer_workspace_bytes(self.cfg, T)
        if self.ws is None or nb > self.ws_bytes:
            self.ws = torch.empty(max(nb, 256), dtype=torch.uint8, device=self.pool.device)
            self.ws_bytes = nb
        return self.ws

    def layer_forward(self, l: int, x: torch.Tensor, y: torch.Tensor, y32=None, idx_out=None, stream=None):
        T = x.shape[0]
        ws = self.workspace(T)
        B.moe_pooled_layer_forward(self.cfg, self.handle, l, self.resident[l]["struct"], x, T, y, y32, idx_out,
                                   ws, self.ws_bytes, stream)

    def table_device(self, l: int) -> torch.Tensor:
        """Copy of layer l's device table row ([E] int32)."""
        ptr, _ = B.slot_pool_layer(self.handle, l)
        return torch.as_tensor(_DeviceArray(ptr, self.E), device=self.pool.device).clone()

    def blob(self, l: int, e: int) -> torch.Tensor:
        """Expert e of layer l as the backing store holds it (CPU bytes)."""
        if self.backing is not None:
            return self.backing[l, e, :self.blob_bytes]
        with open(self.file_path, "rb") as f:
            f.seek((l * self.E + e) * self.file_stride)
            return torch.frombuffer(bytearray(f.read(self.blob_bytes)), dtype=torch.uint8)

    def slot_bytes(self, l: int, slot: int) -> torch.Tensor:
        base = (l * self.S + slot) * self.stride
        return self.pool[base:base + self.blob_bytes]

    def stats(self) -> dict:
        return B.slot_pool_stats(self.handle)

    def close(self):
        if self.handle:
            torch.cuda.synchronize()
            B.slot_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class _DeviceArray:
    """An int32 device array at a raw address, viewable by torch.as_tensor."""

    def __init__(self, ptr: int, n: int):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i4", "data": (ptr, False), "version": 3}
