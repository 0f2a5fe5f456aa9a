"""Oracle of the epoch-level controller: Coordinator, Quant Orchestrator and
Pipeline Adaptor of the SYLVIE guide.

TEST INFRASTRUCTURE ONLY -- imported by tests, never by the library.

Sources (SYLVIE guide, "SYLVIE: 3D-adaptive and Universal System for
Large-scale Graph Neural Network Training"):
  * section 8 (time-dimension adaptivity): the averaged loss L_t over N
    partitions, the exponential moving average F_t = lambda F_{t-1} +
    (1 - lambda) L_t, the loss-descent rate over the epoch time et_t, and the
    four-branch rule for the next base width b_{t+1};
  * section 10 (execution-dimension adaptivity): the Pipeline Adaptor forces
    a synchronous epoch t+1 when LDR_t < LDR_{t-delta}, else runs it
    asynchronously;
  * section 11 (end-to-end pseudocode): start from the smallest width in a
    synchronous mode; for t <= delta the width and the mode are kept.

Readings (listed in the design notes):
  * sign: the formula is printed as (F_t - F_{t-1}) / et_t, yet the text
    calls a smaller LDR worse progress and raises precision on it.  Both hold
    only for the descent rate (F_{t-1} - F_t) / et_t, which is used here.
  * first epoch: F_0 = L_0 (the pseudocode's "initialise on the first
    round") and LDR_0 = 0; LDR_0 is never compared, since a comparison needs
    t > delta >= 1.
  * arithmetic: L_t sums the partition losses in index order and divides by
    N; F_t = (lambda F_{t-1}) + ((1 - lambda) L_t), all IEEE double.
"""
from __future__ import annotations

WIDTHS = (1, 2, 4, 8)


class LdrController:
    """One controller; ``report`` takes an epoch's partition losses and time
    and returns (base width, asynchronous?) for the next epoch."""

    def __init__(self, lam=0.9, delta=5, b_min=1, b_max=8):
        assert 0.0 <= lam < 1.0 and delta >= 1
        assert b_min in WIDTHS and b_max in WIDTHS and b_min <= b_max
        self.lam, self.delta, self.b_min, self.b_max = lam, delta, b_min, b_max
        self.t = 0
        self.b = b_min          # the pseudocode's online initialisation
        self.asynchronous = False
        self.F_prev = None
        self.history = []       # (L_t, F_t, LDR_t, b for t+1, async for t+1)

    def report(self, partition_losses, epoch_seconds):
        assert len(partition_losses) >= 1 and epoch_seconds > 0
        total = 0.0
        for x in partition_losses:          # L_t = sum_n L_t^n / N
            total += float(x)
        L = total / len(partition_losses)
        t = self.t
        if self.F_prev is None:             # first epoch
            F = L
            ldr = 0.0
        else:
            F = self.lam * self.F_prev + (1.0 - self.lam) * L
            ldr = (self.F_prev - F) / epoch_seconds
        if t == 0:
            self.b = self.b_min
        elif t > self.delta:
            past = self.history[t - self.delta][2]
            if ldr < past:                  # descent slowed
                if self.b < self.b_max:
                    self.b = 2 * self.b
                self.asynchronous = False
            else:
                if self.b > self.b_min:
                    self.b = self.b // 2
                self.asynchronous = True
        self.history.append((L, F, ldr, self.b, self.asynchronous))
        self.F_prev = F
        self.t = t + 1
        return self.b, self.asynchronous


def run(losses, times, lam=0.9, delta=5, b_min=1, b_max=8):
    """Feeds a whole sequence of epochs; returns the controller."""
    c = LdrController(lam, delta, b_min, b_max)
    for ls, et in zip(losses, times):
        c.report(ls, et)
    return c
