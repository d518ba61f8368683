"""Expert-health monitor for a serving loop.

Page "Qwen3.5-MoE与Qwen3-MoE架构差异深度解析", section 6, recommends watching two
numbers at the serving gateway: over the last minute, the expert that was
activated least often, and the standard deviation of all experts'
activation counts; when the deviation stays above 20 for five minutes in a
row, raise an alert (abnormal traffic, or a model that has started to lean
on a few experts).

The counts stay on the device: every layer call adds its expert_counts into
an int64 window (moe_expert_counts_accumulate), and closing a window runs
one small kernel (moe_expert_health) and reads back three numbers.  The
windowing and the alert rule are host logic.  When data-parallel ranks each
serve part of the traffic, the gateway's view is the sum over the ranks: with
a process group, closing a window first sums the ranks' windows (one
all-reduce of E int64 counts), so every rank reports the same health.
"""
from __future__ import annotations

import dataclasses
import time
from typing import Callable, List, Optional

import torch

from . import binding as B


@dataclasses.dataclass(frozen=True)
class WindowHealth:
    end: float            # clock value when the window closed
    least_expert: int     # fewest activations (ties: the lower id)
    mean: float           # mean activations per expert
    std: float            # population standard deviation of the activations
    alert: bool           # std above the threshold in this and the previous windows


class ExpertHealthMonitor:
    """Windows of expert activation counts and the alert rule.

    ``record(expert_counts)`` takes a layer call's int32 [E] counts (the
    ``counts`` buffer of ``MoELayer.buffers``) and closes the window once
    ``window_s`` of ``clock`` time have passed since it opened.  An alert is
    raised when the last ``alert_windows`` closed windows all have a
    standard deviation above ``std_threshold``.  ``accumulate`` and
    ``reduce`` default to the library's device entry points.

    For a layer with an expert capacity, the ``counts`` buffer holds the
    assignments each expert kept, never more than the capacity, so an
    overloaded expert shows as a count at the capacity rather than as its
    full demand and the deviation understates the imbalance.  To watch the
    demand of a capped layer, record the per-expert counts of the routed ids
    (``topk_ids``) instead."""

    def __init__(self, E: int, device, window_s: float = 60.0, std_threshold: float = 20.0,
                 alert_windows: int = 5, clock: Callable[[], float] = time.monotonic,
                 accumulate: Optional[Callable] = None, reduce: Optional[Callable] = None,
                 process_group=None):
        if E < 1 or window_s <= 0 or alert_windows < 1:
            raise ValueError("E >= 1, window_s > 0 and alert_windows >= 1 are required")
        self.E = E
        self.window_s = float(window_s)
        self.std_threshold = float(std_threshold)
        self.alert_windows = int(alert_windows)
        self.clock = clock
        self.window = torch.zeros(E, dtype=torch.int64, device=device)
        self._accumulate = accumulate or B.moe_expert_counts_accumulate
        self._reduce = reduce or self._device_reduce
        self.process_group = process_group
        self.history: List[WindowHealth] = []
        self.opened = clock()

    @staticmethod
    def _device_reduce(window):
        least, mean_std = B.moe_expert_health(window)
        ms = mean_std.cpu()
        return int(least.item()), float(ms[0]), float(ms[1])

    @property
    def alert(self) -> bool:
        return bool(self.history) and self.history[-1].alert

    def record(self, expert_counts) -> Optional[WindowHealth]:
        """Add one call's counts; returns the window's health if it closed.
        With a process group windows never close here (the ranks' clocks
        need not agree): every rank calls close_window at the same point."""
        self._accumulate(expert_counts, self.window)
        if self.process_group is None and self.clock() - self.opened >= self.window_s:
            return self.close_window()
        return None

    def window_due(self) -> bool:
        """Whether the open window has lasted window_s on this rank's clock."""
        return self.clock() - self.opened >= self.window_s

    def close_window(self) -> WindowHealth:
        """Reduce the open window (summed over the ranks of the process
        group, if any) and start the next.  With a process group every rank
        must close its windows in the same order."""
        if self.process_group is not None:
            import torch.distributed as dist
            dist.all_reduce(self.window, op=dist.ReduceOp.SUM, group=self.process_group)
        least, mean, std = self._reduce(self.window)
        recent = [h.std for h in self.history[-(self.alert_windows - 1):]] \
            if self.alert_windows > 1 else []
        above = std > self.std_threshold and len(recent) == self.alert_windows - 1 and all(
            s > self.std_threshold for s in recent)
        now = self.clock()
        h = WindowHealth(end=now, least_expert=least, mean=mean, std=std, alert=above)
        self.history.append(h)
        self.window.zero_()
        self.opened = now
        return h
