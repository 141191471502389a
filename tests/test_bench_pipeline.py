"""The end-to-end loop of bench.py (timed_e2e) overlaps the host copies of one
step with the kernels of its neighbours on three streams.  Checked on the CPU
with a recording stand-in for torch.cuda: every operation, event record and
event wait becomes a node of a happens-before graph (stream order plus
record -> wait edges), and every pair of accesses to one buffer of which one
writes must be ordered in it.  Mutants with one of the waits removed must
show a race, so the check is not vacuous."""
import inspect
import itertools
import os
import sys
import textwrap
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class Graph:
    def __init__(self):
        self.succ = []       # node -> successors
        self.access = []     # node -> (reads, writes)

    def node(self, reads=(), writes=()):
        self.succ.append([])
        self.access.append((tuple(reads), tuple(writes)))
        return len(self.succ) - 1

    def edge(self, a, b):
        self.succ[a].append(b)

    def reach(self):
        n = len(self.succ)
        out = [None] * n
        for v in reversed(range(n)):  # edges only go from older to newer nodes
            s = {v}
            for w in self.succ[v]:
                s |= out[w]
            out[v] = s
        return out


class FakeStream:
    def __init__(self, g, name, device="cuda:0"):
        self.g, self.name, self.device, self.last = g, name, device, None

    def _append(self, node):
        if self.last is not None:
            self.g.edge(self.last, node)
        self.last = node
        return node

    def op(self, reads=(), writes=()):
        return self._append(self.g.node(reads, writes))

    def wait_event(self, ev):
        w = self._append(self.g.node())
        if ev.node is not None:
            self.g.edge(ev.node, w)


class FakeEvent:
    def __init__(self, g, enable_timing=False):
        self.g, self.node = g, None

    def record(self, stream):
        self.node = stream._append(self.g.node())

    def elapsed_time(self, other):
        return 1.0


class FakeTensor:
    def __init__(self, cuda, name):
        self.cuda, self.name = cuda, name

    def copy_(self, src, non_blocking=False):
        self.cuda.current.op(reads=(src.name,), writes=(self.name,))
        return self


def fake_torch(g, main):
    cuda = types.SimpleNamespace()
    cuda.current = main
    cuda.Stream = lambda device=None: FakeStream(g, "side", device)
    cuda.Event = lambda enable_timing=False: FakeEvent(g, enable_timing)

    class _Ctx:
        def __init__(self, s):
            self.s = s

        def __enter__(self):
            self.prev, cuda.current = cuda.current, self.s

        def __exit__(self, *a):
            cuda.current = self.prev

    cuda.stream = _Ctx
    cuda.synchronize = lambda: None
    return types.SimpleNamespace(cuda=cuda), cuda


def run_pipeline(fn, n_steps):
    """Run a timed_e2e-like function on fakes; returns the graph, the index
    of the first node it created (the start event's record) and the nodes of
    the compute calls."""
    g = Graph()
    main = FakeStream(g, "main")
    torch, cuda = fake_torch(g, main)
    T = lambda n: FakeTensor(cuda, n)
    h2d = [[(T("in%d.%s" % (b, n)), T("host.%s" % n)) for n in ("Q", "K")] for b in (0, 1)]
    d2h = [[(T("hostout.%s" % n), T("out%d.%s" % (b, n))) for n in ("O", "dQ")] for b in (0, 1)]
    work = []

    def compute(b):
        work.append(main.op(reads=("in%d.Q" % b, "in%d.K" % b),
                            writes=("out%d.O" % b, "out%d.dQ" % b)))

    first = len(g.succ)
    ms = fn(torch, main, h2d, d2h, compute, n_steps)
    assert ms == pytest.approx(1.0 / n_steps)
    return g, first, work


def races(g):
    r = g.reach()
    acc = [(v, set(rd), set(wr)) for v, (rd, wr) in enumerate(g.access) if rd or wr]
    bad = []
    for (a, ra, wa), (b, rb, wb) in itertools.combinations(acc, 2):
        if (wa & (rb | wb)) or (wb & ra):
            if b not in r[a] and a not in r[b]:
                bad.append((a, b, sorted((wa & (rb | wb)) | (wb & ra))))
    return bad


def timed_e2e():
    sys.path.insert(0, ROOT)
    import bench
    return bench.timed_e2e


@pytest.mark.parametrize("n_steps", [2, 3, 4, 10])
def test_pipelined_copies_have_no_buffer_race(n_steps):
    g, first, work = run_pipeline(timed_e2e(), n_steps)
    assert len(work) == n_steps
    assert races(g) == []
    # every node the loop created lies between the start and stop events:
    # the first node is start's record on the main stream, the last the stop
    r = g.reach()
    last = len(g.succ) - 1
    assert all(v in r[first] for v in range(first, last + 1))
    assert all(last in r[v] for v in range(first, last + 1))


def _mutant(line_fragment):
    src = textwrap.dedent(inspect.getsource(timed_e2e()))
    lines = src.splitlines()
    hit = [i for i, l in enumerate(lines) if line_fragment in l]
    assert len(hit) == 1, line_fragment
    indent = lines[hit[0]][: len(lines[hit[0]]) - len(lines[hit[0]].lstrip())]
    lines[hit[0]] = indent + "pass"
    ns = {}
    exec("\n".join(lines), ns)
    return ns["timed_e2e"]


@pytest.mark.parametrize("fragment", [
    "up.wait_event(computed[s - 2])",       # inputs overwritten while still read
    "stream.wait_event(loaded[s])",         # kernels before their inputs arrive
    "stream.wait_event(drained[s - 2])",    # results overwritten before copied out
    "down.wait_event(computed[s])",         # results copied out before written
])
def test_each_wait_is_needed(fragment):
    g, _, _ = run_pipeline(_mutant(fragment), 4)
    assert races(g), fragment


def test_stop_waits_for_the_last_result_copy():
    fn = _mutant("stream.wait_event(drained[n_steps - 1])")
    g, first, _ = run_pipeline(fn, 3)
    r = g.reach()
    last = len(g.succ) - 1
    assert not all(last in r[v] for v in range(first, last + 1))
