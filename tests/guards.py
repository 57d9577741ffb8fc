"""Guard regions around device buffers: the stand-in for a memory checker.

A Guarded buffer is a larger device allocation whose first and last GUARD bytes hold a
fixed byte pattern; `inner` is the 256-byte-aligned region between them that a call writes.
check() fails if any guard byte changed, i.e. if the call wrote outside its array.
"""
import torch

from mla_latent_kv_17_gb300 import ops

GUARD = 4096
HEAD, TAIL = 0xA5, 0x5A


class Guarded:
    def __init__(self, nbytes, device="cuda"):
        self.nbytes = int(nbytes)
        self.full = torch.zeros(self.nbytes + 2 * GUARD, dtype=torch.uint8, device=device)
        self.full[:GUARD] = HEAD
        self.full[GUARD + self.nbytes:] = TAIL
        self.inner = self.full[GUARD:GUARD + self.nbytes]

    def check(self, what=""):
        head = self.full[:GUARD]
        tail = self.full[GUARD + self.nbytes:]
        assert bool((head == HEAD).all()), f"{what}: a write landed in the guard before the array"
        assert bool((tail == TAIL).all()), f"{what}: a write landed in the guard after the array"


def guarded_workspace(B, H, num_sms=0):
    """An ops.Workspace whose buffer sits between guard regions (ws.guard)."""
    ws = ops.Workspace(B, H, num_sms)
    g = Guarded(ws.nbytes, device=ws.buf.device)
    ws.buf = g.inner
    ws.guard = g
    return ws
