"""Tensor-parallel groups: one process per GPU, the ranks' buffers shared
through CUDA IPC.

A ``TPGroup`` gives each rank of a ``torch.distributed`` process group a
[T, H] buffer (where the rank's row-parallel layer writes its partial, and
where y for all T rows appears after the call) and, optionally, a signal pad
for the in-kernel barrier between ranks; it exchanges their IPC handles over
the process group (any backend that carries Python objects, gloo or nccl) and
opens the other ranks' ones, so that every rank addresses every buffer.  The
compute call is ``rarn_tp_reduce_add_rms_norm`` ("Tokenweave fused-RMSNorm-AR
kernel", Code walkthrough: reduce-scatter, residual add + norm, all-gather).

The IPC backend is a parameter so that the exchange and the bookkeeping can be
exercised without a GPU.
"""
from __future__ import annotations

import residual_add_rmsnorm_gb300 as rarn


class NativeIpc:
    """CUDA IPC through the library's rarn_ipc_export / import / close."""

    def export(self, t) -> bytes:
        return rarn.ipc_export(t)

    def open(self, handle: bytes) -> int:
        return rarn.ipc_import(handle)

    def close(self, ptr: int) -> None:
        rarn.ipc_close(ptr)


_TORCH_DTYPES = {"f32": "float32", "f16": "float16", "bf16": "bfloat16"}


class TPGroup:
    """This rank's view of an N-rank tensor-parallel group.

    buffer     this rank's [T, H] buffer (write the partial here)
    buffers    every rank's buffer address, in rank order, as this process
               addresses it (its own buffer's data pointer at its own rank)
    signals    every rank's signal pad address, or None without the barrier
    rows       (r0, r1): the rows this rank owns and keeps the residual of
    """

    def __init__(self, T: int, H: int, dtype: str, device, group=None, signals: bool = True,
                 ipc=None):
        import torch
        import torch.distributed as dist
        self.T, self.H, self.dtype = T, H, dtype
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        if self.world > rarn.TP_MAX_RANKS:
            raise ValueError(f"at most {rarn.TP_MAX_RANKS} ranks")
        self.ipc = ipc if ipc is not None else NativeIpc()
        tdt = getattr(torch, _TORCH_DTYPES[dtype])
        self.buffer = torch.empty((T, H), dtype=tdt, device=device)
        self.pad = (torch.zeros(rarn.TP_SIGNAL_BYTES // 4, dtype=torch.int32, device=device)
                    if signals else None)
        mine = (self.ipc.export(self.buffer),
                self.ipc.export(self.pad) if signals else None)
        handles = [None] * self.world
        dist.all_gather_object(handles, mine, group=group)
        self._opened = []
        self.buffers, sig = [], []
        for q, (hb, hs) in enumerate(handles):
            if q == self.rank:
                self.buffers.append(self.buffer.data_ptr())
                sig.append(self.pad.data_ptr() if signals else None)
                continue
            pb = self.ipc.open(hb)
            self._opened.append(pb)
            self.buffers.append(pb)
            if signals:
                ps = self.ipc.open(hs)
                self._opened.append(ps)
                sig.append(ps)
        self.signals = sig if signals else None
        self.rows = rarn.tp_rows(T, self.world, self.rank)

    def __call__(self, residual, gamma, eps: float) -> None:
        """Reduce-scatter, residual add + norm, all-gather: afterwards this
        rank's ``buffer`` holds y for all T rows (once every rank's call has
        completed, which the signal pads ensure before the call returns on the
        stream; without them the caller orders the ranks)."""
        rarn.tp_reduce_add_rms_norm(self.buffers, self.rank, residual, gamma, eps, self.T,
                                    signals=self.signals)

    def close(self) -> None:
        """Release the other ranks' mappings (this rank's memory stays)."""
        while self._opened:
            self.ipc.close(self._opened.pop())
