"""Host logic of the bench's device-timed loop, on CPU.

The timed loops keep a bounded number of step graphs in flight: replay i is enqueued
only once replay i - in_flight has finished, which the loop learns from an event it
recorded right after that replay.  A stand-in event class records the order of
replays, records and waits, so the bound can be checked without a GPU.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


class _Log:
    def __init__(self):
        self.ops = []


class _Graph:
    def __init__(self, log, i):
        self.log, self.i = log, i

    def replay(self):
        self.log.ops.append(("replay", self.i))


def _fake_events(log, monkeypatch):
    created = []

    class Event:
        def __init__(self, *a, **k):
            self.id = len(created)
            self.last = None                   # index of the replay recorded after
            created.append(self)

        def record(self, *a):
            self.last = log.replay_count
            log.ops.append(("record", self.id, self.last))

        def synchronize(self):
            log.ops.append(("wait", self.id, self.last))

    monkeypatch.setattr(bench.torch.cuda, "Event", Event)
    return created


@pytest.mark.parametrize("n, in_flight", [(0, 8), (1, 8), (5, 8), (8, 8), (9, 8), (50, 8), (7, 2), (30, 1)])
def test_replays_in_order_with_at_most_in_flight_pending(monkeypatch, n, in_flight):
    log = _Log()
    log.replay_count = 0
    _fake_events(log, monkeypatch)

    def graph_of(i):
        g = _Graph(log, i)
        orig = g.replay

        def replay():
            orig()
            log.replay_count += 1
        g.replay = replay
        return g

    bench.replay_in_flight(graph_of, n, in_flight=in_flight)
    replays = [op[1] for op in log.ops if op[0] == "replay"]
    assert replays == list(range(n))
    # when replay i is enqueued, at most in_flight - 1 earlier replays are not yet known
    # to have finished (a wait on the event recorded after replay k shows k + 1 done)
    done = 0
    for op in log.ops:
        if op[0] == "wait":
            done = max(done, op[2])
        elif op[0] == "replay":
            assert op[1] - done <= in_flight - 1, (op[1], done)
    # and the loop waits no more than that: replay in_flight + k waits only for replay k
    waits = [op for op in log.ops if op[0] == "wait"]
    assert len(waits) == max(0, n - in_flight)
    for k, w in enumerate(waits):
        assert w[2] == k + 1


def test_default_bound_is_eight():
    assert bench.IN_FLIGHT == 8
