"""Upload a generated layer to the GPU.

Draws every tensor of a LayerConfig with the counter-based generator on the
host, copies it to the device and packs the expert weights there with the
library's moe_pack_w4 (or, with fmt="w8", moe_pack_w8: E4M3 codes and one fp32
scale per row).  Holds no layer arithmetic of its own.  An optional
``on_expert(e, w_gateup, w_down)`` callback sees each expert's fp32 weights on
the host (e = -1 for the shared expert) so a caller can quantise the same
values another way without drawing them twice.
"""
from __future__ import annotations

import queue
import threading
from dataclasses import dataclass, field

import numpy as np
import torch

from . import LayerConfig, gen_down, gen_gateup, gen_router, gen_x


@dataclass
class DeviceLayer:
    cfg: LayerConfig
    x: torch.Tensor          # bf16 bits as int16 [T][d] (batch 0)
    W_r: torch.Tensor        # fp32 [E][d]
    bias: torch.Tensor       # fp32 [E]
    gu_q: torch.Tensor       # uint8 [E][2F][d/2]           (w8: [E][2F][d] codes)
    gu_s: torch.Tensor       # int16 (fp16 bits) [E][2F][d/g] (w8: fp32 [E][2F])
    dn_q: torch.Tensor       # uint8 [E][d][F/2]            (w8: [E][d][F])
    dn_s: torch.Tensor       # int16 [E][d][F/g]            (w8: fp32 [E][d])
    sgu_q: torch.Tensor      # shared gate+up
    sgu_s: torch.Tensor
    sdn_q: torch.Tensor      # shared down
    sdn_s: torch.Tensor
    x_batches: list = field(default_factory=list)  # extra activation batches
    fmt: str = "w4"

    def dims(self, flags: int = 0, T: int | None = None):
        import moe_expert_layer_sigmoid_gb300 as moe
        c = self.cfg
        return moe.Dims(T=c.T if T is None else T, d=c.d, E=c.E, k=c.k, F=c.F, F_s=c.Fs,
                        group=c.group, flags=flags)

    def w8s(self):
        import moe_expert_layer_sigmoid_gb300 as moe
        assert self.fmt == "w8"
        return (moe.w8(self.gu_q, self.gu_s), moe.w8(self.dn_q, self.dn_s),
                moe.w8(self.sgu_q, self.sgu_s), moe.w8(self.sdn_q, self.sdn_s))

    def w4s(self):
        import moe_expert_layer_sigmoid_gb300 as moe
        assert self.fmt == "w4"
        return (moe.w4(self.gu_q, self.gu_s), moe.w4(self.dn_q, self.dn_s),
                moe.w4(self.sgu_q, self.sgu_s), moe.w4(self.sdn_q, self.sdn_s))

    def packed_bytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (
            self.gu_q, self.gu_s, self.dn_q, self.dn_s, self.sgu_q, self.sgu_s, self.sdn_q,
            self.sdn_s))


def _x_tensor(cfg, batch, device):
    return torch.from_numpy(gen_x(cfg, batch).view(np.int16)).to(device)


def upload(cfg: LayerConfig, device="cuda", extra_batches: int = 0, on_expert=None,
           prefetch: int = 3, fmt: str = "w4") -> DeviceLayer:
    import moe_expert_layer_sigmoid_gb300 as moe

    E, F, Fs, d, g = cfg.E, cfg.F, cfg.Fs, cfg.d, cfg.group
    wr, b = gen_router(cfg)
    u8 = dict(dtype=torch.uint8, device=device)
    if fmt == "w8":
        f32 = dict(dtype=torch.float32, device=device)
        gu_q, gu_s = torch.empty((E, 2 * F, d), **u8), torch.empty((E, 2 * F), **f32)
        dn_q, dn_s = torch.empty((E, d, F), **u8), torch.empty((E, d), **f32)
        sgu_q, sgu_s = torch.empty((2 * Fs, d), **u8), torch.empty(2 * Fs, **f32)
        sdn_q, sdn_s = torch.empty((d, Fs), **u8), torch.empty(d, **f32)
        pack = lambda w, q, s, stream: moe.moe_pack_w8(w, q, s, stream=stream)
    else:
        i16 = dict(dtype=torch.int16, device=device)
        gu_q, gu_s = torch.empty((E, 2 * F, d // 2), **u8), torch.empty((E, 2 * F, d // g), **i16)
        dn_q, dn_s = torch.empty((E, d, F // 2), **u8), torch.empty((E, d, F // g), **i16)
        sgu_q, sgu_s = torch.empty((2 * Fs, d // 2), **u8), torch.empty((2 * Fs, d // g), **i16)
        sdn_q, sdn_s = torch.empty((d, Fs // 2), **u8), torch.empty((d, Fs // g), **i16)
        pack = lambda w, q, s, stream: moe.moe_pack_w4(w, g, q, s, stream=stream)

    # host producer: draw expert weights ahead of the device packing
    work: queue.Queue = queue.Queue(maxsize=prefetch)

    def produce():
        try:
            for e in list(range(E)) + [-1]:
                work.put((e, gen_gateup(cfg, e), gen_down(cfg, e)))
        except BaseException as exc:  # surface in the consumer
            work.put(exc)
            return
        work.put(None)

    th = threading.Thread(target=produce, daemon=True)
    th.start()
    stream = torch.cuda.current_stream(device)
    while True:
        item = work.get()
        if item is None:
            break
        if isinstance(item, BaseException):
            raise item
        e, wgu, wdn = item
        if on_expert is not None:
            on_expert(e, wgu, wdn)
        wgu_d = torch.from_numpy(wgu).to(device)
        wdn_d = torch.from_numpy(wdn).to(device)
        if e >= 0:
            pack(wgu_d, gu_q[e], gu_s[e], stream)
            pack(wdn_d, dn_q[e], dn_s[e], stream)
        else:
            pack(wgu_d, sgu_q, sgu_s, stream)
            pack(wdn_d, sdn_q, sdn_s, stream)
    th.join()
    torch.cuda.synchronize(device)
    layer = DeviceLayer(
        cfg=cfg, x=_x_tensor(cfg, 0, device), W_r=torch.from_numpy(wr).to(device),
        bias=torch.from_numpy(b).to(device), gu_q=gu_q, gu_s=gu_s, dn_q=dn_q, dn_s=dn_s,
        sgu_q=sgu_q, sgu_s=sgu_s, sdn_q=sdn_q, sdn_s=sdn_s, fmt=fmt)
    layer.x_batches = [_x_tensor(cfg, bi, device) for bi in range(1, 1 + extra_batches)]
    return layer
