"""Device storage of one MoE layer and its strata_moe_layer descriptor.

Holds torch tensors (torch is used for device memory and streams only) and
fills the C struct with their addresses. Expert weights arrive as fp16 host
arrays and are quantized on the device by strata_quantize_groups_bits (4-bit
codes, two per byte, by default; 8-bit codes, one per byte, with bits=8).
"""
from __future__ import annotations

import ctypes

from . import (GROUP, StrataError, check, ptr, strata_moe_layer, strata_moe_workspace_size,
               strata_quantize_groups_bits, strata_read_status)


class MoELayer:
    def __init__(self, H: int, I: int, E: int, k: int, shared: int, flags: int = 0,
                 device: str = "cuda", group: int = GROUP, bits: int = 4):
        import torch
        self.H, self.I, self.E, self.k, self.shared, self.flags = H, I, E, k, shared, flags
        self.group = group
        self.bits = bits
        per = 8 // bits  # codes per byte
        self.device = torch.device(device)
        n = E + shared
        u8, f16, f32 = torch.uint8, torch.float16, torch.float32
        self.w_router = torch.zeros(E, H, dtype=f32, device=self.device)
        self.bias = None
        self.gate_codes = torch.zeros(n, I, H // per, dtype=u8, device=self.device)
        self.gate_scales = torch.zeros(n, I, H // group, dtype=f16, device=self.device)
        self.up_codes = torch.zeros(n, I, H // per, dtype=u8, device=self.device)
        self.up_scales = torch.zeros(n, I, H // group, dtype=f16, device=self.device)
        self.down_codes = torch.zeros(n, H, I // per, dtype=u8, device=self.device)
        self.down_scales = torch.zeros(n, H, I // group, dtype=f16, device=self.device)
        self._status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self._stage = None

    # ---------------------------------------------------------------- weights
    def set_router(self, w_router, bias=None, fp16: bool = False):
        """Router weights [E,H]: fp32, or stored as fp16 (STRATA_ROUTER_FP16) when fp16=True."""
        import torch
        from . import STRATA_ROUTER_FP16
        if fp16:
            self.w_router = torch.as_tensor(w_router).to(torch.float16).to(self.device)
            self.flags |= STRATA_ROUTER_FP16
        else:
            self.w_router = torch.as_tensor(w_router, dtype=torch.float32).to(self.device)
            self.flags &= ~STRATA_ROUTER_FP16
        self.bias = None if bias is None else torch.as_tensor(bias, dtype=torch.float32).to(self.device)

    def load_expert_fp16(self, e: int, gate, up, down, stream=None):
        """Upload fp16 [I,H], [I,H], [H,I] host arrays and quantize them into expert slot e."""
        import torch
        mats = [(gate, self.gate_codes, self.gate_scales), (up, self.up_codes, self.up_scales),
                (down, self.down_codes, self.down_scales)]
        for w, codes, scales in mats:
            src = torch.from_numpy(w) if not isinstance(w, torch.Tensor) else w
            n_el = src.numel()
            if self._stage is None or self._stage.numel() < n_el:
                self._stage = torch.empty(n_el, dtype=torch.float16, device=self.device)
            dst = self._stage[:n_el].view(src.shape)
            dst.copy_(src, non_blocking=False)
            rows, cols = src.shape
            check(strata_quantize_groups_bits(dst, rows, cols, codes[e], scales[e], self._status,
                                              group_size=self.group, bits=self.bits,
                                              stream=stream),
                  "strata_quantize_groups_bits")

    def check_status(self, stream=None):
        st, v = strata_read_status(self._status, stream)
        if st != 0:
            raise StrataError(st, f"quantize device status 0x{v:x}")

    def copy_expert_from(self, other: "MoELayer"):
        """Take another layer's quantized experts (same shapes)."""
        for name in ("gate_codes", "gate_scales", "up_codes", "up_scales", "down_codes",
                     "down_scales"):
            getattr(self, name).copy_(getattr(other, name))

    # ---------------------------------------------------------------- C descriptor
    def struct(self) -> strata_moe_layer:
        s = strata_moe_layer()
        s.H, s.I, s.E, s.k = self.H, self.I, self.E, self.k
        s.has_shared, s.flags = self.shared, self.flags
        s.w_router = ptr(self.w_router)
        s.bias = ptr(self.bias)
        s.gate_codes, s.gate_scales = ptr(self.gate_codes), ptr(self.gate_scales)
        s.up_codes, s.up_scales = ptr(self.up_codes), ptr(self.up_scales)
        s.down_codes, s.down_scales = ptr(self.down_codes), ptr(self.down_scales)
        s.group_size = self.group
        s.bits = self.bits
        return s

    def workspace_size(self, T_max: int) -> int:
        return strata_moe_workspace_size(self.struct(), T_max)

    def expert_bytes(self) -> int:
        n = 3 * self.H * self.I
        return n * self.bits // 8 + 2 * (n // self.group)


__all__ = ["MoELayer", "ctypes"]
