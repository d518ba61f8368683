"""Host logic of the expert-health monitor (windows and the alert rule of
page [B] section 6), with the window arithmetic done on the CPU by the
oracle in place of the device kernels."""
import numpy as np
import pytest
import torch

import oracle
from sparse_moe_expert_gb300.health import ExpertHealthMonitor


class FakeClock:
    def __init__(self):
        self.t = 0.0

    def __call__(self):
        return self.t


def cpu_monitor(E, clock, **kw):
    def accumulate(counts, window):
        window += counts.to(torch.int64)

    def reduce(window):
        return oracle.expert_health(window.numpy())

    return ExpertHealthMonitor(E, "cpu", clock=clock, accumulate=accumulate, reduce=reduce, **kw)


def counts_with_std(E, std):
    """Counts of E (even) experts whose population std is exactly `std`."""
    return torch.tensor([100 - std, 100 + std] * (E // 2), dtype=torch.int32)


def test_windows_close_after_their_length_and_sum_the_calls():
    clock = FakeClock()
    mon = cpu_monitor(4, clock)
    calls = [torch.tensor(v, dtype=torch.int32) for v in ([1, 2, 3, 0], [0, 2, 1, 5], [4, 0, 0, 1])]
    for i, c in enumerate(calls):
        clock.t = 20.0 * i
        assert mon.record(c) is None
    clock.t = 60.0
    h = mon.record(torch.zeros(4, dtype=torch.int32))
    total = np.sum([c.numpy() for c in calls], axis=0)
    assert (h.least_expert, h.mean, h.std) == oracle.expert_health(total)
    assert h.end == 60.0 and not h.alert
    assert int(mon.window.sum()) == 0 and mon.opened == 60.0


@pytest.mark.parametrize("windows", [5, 3])
def test_alert_after_consecutive_windows_above_threshold(windows):
    clock = FakeClock()
    mon = cpu_monitor(8, clock, alert_windows=windows)
    flags = []
    for i in range(windows + 2):
        clock.t = 60.0 * (i + 1)
        h = mon.record(counts_with_std(8, 21))
        flags.append(h.alert)
    # the alert starts with the windows-th window above 20 and stays
    assert flags == [False] * (windows - 1) + [True] * 3
    # one window at or below the threshold clears it and restarts the count
    clock.t += 60.0
    assert mon.record(counts_with_std(8, 20)).alert is False
    for i in range(windows - 1):
        clock.t += 60.0
        assert mon.record(counts_with_std(8, 25)).alert is False
    clock.t += 60.0
    assert mon.record(counts_with_std(8, 25)).alert is True
    assert mon.alert


def test_least_expert_tracks_the_quietest_expert():
    clock = FakeClock()
    mon = cpu_monitor(6, clock, window_s=10.0)
    clock.t = 10.0
    h = mon.record(torch.tensor([5, 5, 3, 3, 9, 7], dtype=torch.int32))
    assert h.least_expert == 2


def test_monitor_arguments():
    with pytest.raises(ValueError):
        cpu_monitor(0, FakeClock())
    with pytest.raises(ValueError):
        cpu_monitor(4, FakeClock(), window_s=0)
