"""Stream / event ordering of pipeline.HostPipeline, checked on the CPU with
recording stand-ins for CUDA streams, events and the step itself: a device
slot is refilled only after the step that last used it has run, and is run
again only after its previous results have been copied out."""
import torch

import sparse_causal_flash_gb300.pipeline as pl


class FakeEvent:
    n = 0

    def __init__(self, *a, **k):
        FakeEvent.n += 1
        self.name = f"ev{FakeEvent.n}"

    def record(self, stream):
        stream.log.append(("record", self.name))


class FakeStream:
    def __init__(self, name, log):
        self.name, self.log = name, log

    def wait_event(self, ev):
        self.log.append((self.name, "wait", ev.name))

    def wait_stream(self, other):
        self.log.append((self.name, "wait_stream", other.name))


class FakeStep:
    def __init__(self, *a, **k):
        z = torch.zeros(1)
        self.o = self.lse = self.dq = self.dk = self.dv = z

    def run(self, *a, stream=None, **k):
        stream.log.append((stream.name, "run", id(self)))


def test_slots_alternate_and_wait_for_reuse(monkeypatch):
    log = []
    streams = iter([FakeStream("h2d", log), FakeStream("d2h", log)])
    main = FakeStream("main", log)
    monkeypatch.setattr(pl, "Step", FakeStep)
    monkeypatch.setattr(pl.torch.cuda, "Stream", lambda *a, **k: next(streams))
    monkeypatch.setattr(pl.torch.cuda, "Event", FakeEvent)

    class Ctx:
        def __init__(self, s):
            pass

        def __enter__(self):
            return self

        def __exit__(self, *a):
            return False

    monkeypatch.setattr(pl.torch.cuda, "stream", Ctx)
    monkeypatch.setattr(torch.Tensor, "copy_", lambda self, src, non_blocking=False: self)
    monkeypatch.setattr(pl.torch, "empty", lambda shape, dtype=None, device=None: torch.zeros(shape, dtype=dtype))
    pipe = pl.HostPipeline(2, 1, 1, 4, 4, 64, n_buckets=4, device="cpu")
    hin = {"q": torch.zeros(2), "k": torch.zeros(2), "v": torch.zeros(2), "do": torch.zeros(2), "R": torch.zeros(2)}
    hout = [torch.zeros(1)] * 5
    runs = []
    for _ in range(3):
        runs.append(pipe.submit(hin, hout, 0.125, stream=main))
    # slots alternate: steps 0 and 2 share a Step, step 1 uses the other
    assert runs[0] is runs[2] and runs[0] is not runs[1]
    ev = lambda lst, s: lst[s].name
    first = log[:log.index(("main", "run", id(runs[0])))]
    # no waits on reuse events before a slot was used
    assert not any(e[1] == "wait" and e[2] in (ev(pipe.computed, 0), ev(pipe.drained, 0)) for e in first)
    third = log[log.index(("main", "run", id(runs[1]))):]
    # third submit: h2d waits for slot 0's step, main for slot 0's download
    assert ("h2d", "wait", ev(pipe.computed, 0)) in third
    assert ("main", "wait", ev(pipe.drained, 0)) in third
    i_wait = third.index(("main", "wait", ev(pipe.drained, 0)))
    i_run = [i for i, e in enumerate(third) if e == ("main", "run", id(runs[2]))][0]
    assert i_wait < i_run
    # every step's upload is waited for by the compute stream, every download follows its step
    assert log.count(("main", "wait", ev(pipe.in_ready, 0))) == 2
    assert log.count(("d2h", "wait", ev(pipe.computed, 1))) == 1
