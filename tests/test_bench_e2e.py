"""Host logic of the bench's end-to-end loop (bench.pipelined_e2e): with a fake
torch that records every copy, call and event as a node of a dependency graph
(stream order plus event waits), check that each step's call depends on its own
input copies, each result read depends on its call, an input buffer is
overwritten only after the call two steps back has read it, an output buffer is
reused only after the read two steps back, and the closing event depends on
everything.  No GPU."""

import contextlib
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


class _Graph:
    def __init__(self):
        self.nodes = []  # (kind, info, deps)

    def add(self, kind, info, deps):
        self.nodes.append((kind, info, set(d for d in deps if d is not None)))
        return len(self.nodes) - 1

    def reaches(self, src, dst):
        """True when node dst depends (transitively) on node src."""
        todo, seen = [dst], set()
        while todo:
            n = todo.pop()
            if n == src:
                return True
            if n in seen:
                continue
            seen.add(n)
            todo.extend(self.nodes[n][2])
        return False


class _FakeTorch:
    def __init__(self):
        g = self.graph = _Graph()
        outer = self

        class Stream:
            def __init__(self):
                self.last, self.waits = None, []

            def op(self, kind, info):
                n = g.add(kind, info, [self.last] + self.waits)
                self.last, self.waits = n, []
                return n

            def wait_event(self, ev):
                self.waits.append(ev.node)

            def wait_stream(self, other):
                self.waits.append(other.last)

        class Event:
            def __init__(self, enable_timing=False):
                self.node = None

            def record(self, stream=None):
                s = stream if stream is not None else outer.cur
                self.node = s.op("event", None)

            def elapsed_time(self, other):
                return 1.0

        class Cuda:
            pass

        cuda = Cuda()
        cuda.Stream, cuda.Event = Stream, Event
        cuda.synchronize = lambda: None

        @contextlib.contextmanager
        def stream_ctx(s):
            prev, outer.cur = outer.cur, s
            try:
                yield
            finally:
                outer.cur = prev

        cuda.stream = stream_ctx
        cuda.current_stream = lambda: outer.cur
        self.cuda = cuda
        self.compute = Stream()
        self.cur = self.compute


class _Tensor:
    def __init__(self, torch, name):
        self.torch, self.name = torch, name

    def copy_(self, src, non_blocking=False):
        self.torch.cur.op("copy", (src.name, self.name))


@pytest.mark.parametrize("steps", [1, 2, 3, 7])
def test_pipelined_copies_and_calls_are_ordered(steps):
    t = _FakeTorch()
    g = t.graph
    h_in = [_Tensor(t, "h_q"), _Tensor(t, "h_p")]
    dev_in = [[_Tensor(t, f"q{i}"), _Tensor(t, f"p{i}")] for i in range(2)]
    h_out = _Tensor(t, "h_out")
    dev_out = [_Tensor(t, f"o{i}") for i in range(2)]
    calls = []

    def run(ins, out):
        calls.append(t.compute.op("call", (len(calls), ins[0].name, out.name)))

    ms = bench.pipelined_e2e(t, t.compute, steps, h_in, dev_in, h_out, dev_out, run)
    assert ms == 1.0 / steps and len(calls) == steps
    copies = [(n, info) for n, (kind, info, _) in enumerate(g.nodes) if kind == "copy"]
    end = max(n for n, (kind, _, _) in enumerate(g.nodes) if kind == "event")
    for k, c in enumerate(calls):
        i = k % 2
        assert g.nodes[c][1] == (k, f"q{i}", f"o{i}")
        # this step's input copies: the latest copies into buffer i issued before the call
        ins = [n for n, (src, dst) in copies if dst in (f"q{i}", f"p{i}") and n < c]
        mine = sorted(ins)[-2:]
        assert len(mine) == 2 and all(g.reaches(n, c) for n in mine)
        # its result read: the first copy out of o{i} after the call
        reads = [n for n, (src, dst) in copies if src == f"o{i}" and n > c]
        assert reads and g.reaches(c, reads[0]) and g.reaches(reads[0], end)
        if k + 2 < steps:
            # the inputs of step k + 2 overwrite buffer i only after this call has read it
            later = [n for n, (src, dst) in copies if dst == f"q{i}" and n > c]
            assert later and g.reaches(c, later[0])
            # and step k + 2 writes o{i} only after this step's result was read back
            assert g.reaches(reads[0], calls[k + 2])
    assert all(g.reaches(n, end) for n, _ in copies)
