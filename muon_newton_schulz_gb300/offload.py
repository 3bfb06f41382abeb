"""Muon step on optimizer state kept in host (Grace) memory.

The pages keep state off the GPU when HBM is short: activations are
offloaded to Grace memory over NVLink-C2C ("Training a 1T-Params MoE on EU
public infrastructure", tanhow.com, activation-offload paragraph).  Here the
weights, gradients and momentum (any subset of them) live in host memory and
the library's ``muon_step_host`` runs the step in chunks of whole matrices
through a ring of device staging slots: copies in, ``muon_step`` on the
chunk, copies out, on three streams the library owns, so that the copies of
one chunk overlap the step of another.  This module only builds descriptors
from torch tensors and owns the device workspace (torch provides memory and
the stream).
"""
from __future__ import annotations

import torch

from . import binding as B


class HostOffloadedMuon:
    """Pipelined Muon steps over host-resident tensors.

    ``host_buffers`` selects which of W, G, M (and O, when given) are host
    tensors (``binding.MUON_HOST_*`` bits; default W, G and M); the others are
    device tensors used in place.  ``chunk`` matrices per staging slot,
    ``slots`` slots in the ring."""

    def __init__(self, device: int = 0, chunk: int = 1, slots: int = 3,
                 host_buffers: int = B.MUON_HOST_W | B.MUON_HOST_G | B.MUON_HOST_M, **cfg):
        self.dev = torch.device("cuda", device)
        self.muon = B.MuonStep(device, **cfg)
        self.pl = B.make_pipeline(host_buffers, chunk, slots)
        self._ws = None

    def close(self):
        self.muon.close()

    def workspace_bytes(self, descs, n) -> int:
        st, nbytes = B.muon_host_workspace_size(self.muon.h, descs, n, self.pl)
        if st != B.MUON_OK:
            raise B.MuonError(st, B.muon_last_error_message(self.muon.h))
        return nbytes

    def step(self, Ws, Gs, Ms, lrs, Os=None, sync: bool = True):
        """One step; host tensors among Ws, Ms (and Os) are updated in place.
        With ``sync`` the call returns once the last copy back has completed."""
        descs, n = B.MuonStep.descs_from_tensors(Ws, Gs, Ms, lrs, Os)
        nbytes = self.workspace_bytes(descs, n)
        if self._ws is None or self._ws.numel() < nbytes:
            self._ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.dev)
        stream = torch.cuda.current_stream(self.dev)
        st = B.muon_step_host(self.muon.h, descs, n, self.pl, self._ws.data_ptr(), self._ws.numel(),
                              stream.cuda_stream)
        if st != B.MUON_OK:
            raise B.MuonError(st, B.muon_last_error_message(self.muon.h))
        if sync:
            stream.synchronize()

    def check_status(self):
        """Reads and clears the status words of the last step's chunks (one per
        staging slot) after synchronising the current stream."""
        if self._ws is None:
            return B.MUON_OK
        stream = torch.cuda.current_stream(self.dev).cuda_stream
        return B.muon_check_status(self.muon.h, self._ws.data_ptr(), stream)
