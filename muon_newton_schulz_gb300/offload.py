"""Muon step on optimizer state kept in host (Grace) memory.

The pages keep state off the GPU when HBM is short: activations are
offloaded to Grace memory over NVLink-C2C ("Training a 1T-Params MoE on EU
public infrastructure", tanhow.com, activation-offload paragraph).  Here the
weights, gradients and momentum live in pinned host memory and the step runs
in chunks of whole matrices through a ring of device slots on three streams:
copy in (H2D), ``muon_step`` on the chunk, copy out (D2H) of W and M.  The
copies of one chunk overlap the step of another, so the time approaches the
larger of the transfer time and the compute time.

Only copies and launches are orchestrated here; the step itself is the
library's ``muon_step`` (torch provides device memory, streams and events).
"""
from __future__ import annotations

import torch

from . import binding as B


class HostOffloadedMuon:
    """Pipelined Muon steps over host-resident (pinned) W, G, M lists.

    ``chunk`` matrices per slot, ``slots`` device slots in the ring.  The
    matrices of a call must fit the slot buffers allocated on first use (they
    are re-allocated when a call needs more)."""

    def __init__(self, device: int = 0, chunk: int = 4, slots: int = 3, **cfg):
        self.dev = torch.device("cuda", device)
        self.chunk = max(1, int(chunk))
        self.nslots = max(2, int(slots))
        self.muon = [B.MuonStep(device, **cfg) for _ in range(self.nslots)]
        self.s_in = torch.cuda.Stream(self.dev)
        self.s_run = torch.cuda.Stream(self.dev)
        self.s_out = torch.cuda.Stream(self.dev)
        self._slots = None
        self._shapes = None

    def close(self):
        for m in self.muon:
            m.close()

    def _alloc(self, Wh, Gh, Mh):
        """Chunk list of this batch; slot state is rebuilt when the batch's
        shapes change (device buffers are then created on first use)."""
        n = len(Wh)
        chunks = [list(range(i, min(n, i + self.chunk))) for i in range(0, n, self.chunk)]
        key = (tuple((tuple(w.shape), w.dtype) for w in Wh), self.chunk)
        if self._shapes == key:
            return chunks
        self._slots = []
        for _ in range(self.nslots):
            self._slots.append({
                "done": torch.cuda.Event(),     # D2H of the slot's last chunk finished
                "bufs": {},
            })
        self._shapes = key
        return chunks

    def _slot_tensors(self, slot, idx, Wh):
        """Per-slot device tensors keyed by position in the chunk and shape."""
        out = []
        for k, i in enumerate(idx):
            key = (k, tuple(Wh[i].shape), Wh[i].dtype)
            t = slot["bufs"].get(key)
            if t is None:
                shape = tuple(Wh[i].shape)
                t = (torch.empty(shape, dtype=Wh[i].dtype, device=self.dev),
                     torch.empty(shape, dtype=torch.float32, device=self.dev),
                     torch.empty(shape, dtype=torch.float32, device=self.dev))
                slot["bufs"][key] = t
            out.append(t)
        return out

    def step(self, Wh, Gh, Mh, lrs):
        """One step; Wh and Mh (pinned host tensors) are updated in place.
        Returns when the last copy back has completed."""
        chunks = self._alloc(Wh, Gh, Mh)
        cur = torch.cuda.current_stream(self.dev)
        self.s_in.wait_stream(cur)
        for ci, idx in enumerate(chunks):
            sl = ci % self.nslots
            slot = self._slots[sl]
            dev = self._slot_tensors(slot, idx, Wh)
            # the slot is free once its previous chunk has been copied out
            self.s_in.wait_event(slot["done"])
            with torch.cuda.stream(self.s_in):
                for (w, g, m), i in zip(dev, idx):
                    w.copy_(Wh[i], non_blocking=True)
                    g.copy_(Gh[i], non_blocking=True)
                    m.copy_(Mh[i], non_blocking=True)
                loaded = torch.cuda.Event()
                loaded.record(self.s_in)
            self.s_run.wait_event(loaded)
            with torch.cuda.stream(self.s_run):
                self.muon[sl].step([d[0] for d in dev], [d[1] for d in dev], [d[2] for d in dev],
                                   [lrs[i] for i in idx], stream=self.s_run.cuda_stream)
                stepped = torch.cuda.Event()
                stepped.record(self.s_run)
            self.s_out.wait_event(stepped)
            with torch.cuda.stream(self.s_out):
                for (w, g, m), i in zip(dev, idx):
                    Wh[i].copy_(w, non_blocking=True)
                    Mh[i].copy_(m, non_blocking=True)
                slot["done"].record(self.s_out)
        self.s_out.synchronize()
