"""Helpers for the GPU parity tests: device copies of the seeded inputs and the decision
comparison rule.

Parity rule for decisions (accept lengths, tokens, ancestors, resample flags, lengths): the
GPU must equal the oracle except where the oracle's margin for that decision (distance of the
uniform, or of the compared statistic, to the decision boundary) is below 1e-5; such excused
mismatches are counted and must stay below 1e-4 of the decisions compared. Log-weights and
log-normalisers must agree within 1e-4 absolute.
"""
import numpy as np
import torch

EXCUSE_MARGIN = 1e-5
MAX_EXCUSED_RATE = 1e-4
FLOAT_ATOL = 1e-4


def dev_logits(a: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bits or float32 numpy -> device tensor of the same bytes."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


class DecisionLedger:
    """Counts compared decisions and excused mismatches across a test."""

    def __init__(self):
        self.total = 0
        self.excused = 0
        self.near = 0

    def compare(self, name, got, want, margin):
        got = np.asarray(got).reshape(-1)
        want = np.asarray(want).reshape(-1)
        margin = np.asarray(margin, dtype=np.float64).reshape(-1)
        assert got.shape == want.shape == margin.shape, name
        mism = got != want
        hard = mism & ~(margin < EXCUSE_MARGIN)
        assert not hard.any(), (
            f"{name}: {int(hard.sum())} mismatches with margin >= {EXCUSE_MARGIN} at "
            f"{np.nonzero(hard)[0][:8]} got {got[hard][:8]} want {want[hard][:8]} "
            f"margins {margin[hard][:8]}")
        self.total += got.size
        self.excused += int(mism.sum())
        self.near += int((margin < EXCUSE_MARGIN).sum())

    def finish(self):
        allowed = int(np.floor(MAX_EXCUSED_RATE * max(self.total, 1)))
        assert self.excused <= allowed, (
            f"{self.excused} excused mismatches in {self.total} decisions (allowed {allowed})")
