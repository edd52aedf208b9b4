"""Continuous batching, host side (no GPU): `engine.Batcher` over a fake
engine that keeps sequence lengths and returns as next token the input token
+ 1.  Pinned: requests join at the first step at or after their arrival that
has room (at most max_batch rows per launch), each launch gets every active
sequence at its current length, a request returns exactly max_new tokens (the
prefill's token is the first), its pages are released the step it finishes,
and the finish step is the step of its last decode launch."""
import torch

from moe_decode_megakernel_persistent_gb300.engine import Batcher, Request


class FakeEngine:
    out_device = torch.device("cpu")

    def __init__(self, max_batch):
        self.max_batch = max_batch
        self.length = {}
        self.launches = []     # (step seq ids, positions)
        self.released = []

    def prefill(self, seq_id, prompt, **kw):
        assert seq_id not in self.length
        self.length[seq_id] = int(prompt.numel())
        return torch.tensor([int(prompt[-1]) + 1], dtype=torch.int32)

    def seq_length(self, seq_id):
        return self.length[seq_id]

    def decode_step(self, ids, toks, positions, out):
        assert len(ids) <= self.max_batch and len(set(ids)) == len(ids)
        assert positions == [self.length[i] for i in ids]
        self.launches.append((list(ids), list(positions)))
        out.copy_(toks + 1)
        for i in ids:
            self.length[i] += 1

    def release(self, seq_id):
        self.released.append((seq_id, len(self.launches)))
        del self.length[seq_id]


def _req(sid, n, max_new, arrival):
    return Request(seq_id=sid, prompt=torch.full((n,), 100 * sid, dtype=torch.int32), max_new=max_new,
                   arrival=arrival)


def test_arrivals_batch_cap_tokens_and_finish_steps():
    e = FakeEngine(max_batch=3)
    reqs = [_req(0, 10, 3, 0), _req(1, 20, 2, 0), _req(2, 5, 4, 1), _req(3, 7, 1, 1), _req(4, 9, 5, 1),
            _req(5, 3, 2, 6)]
    out = Batcher(e).run(reqs)
    # every request returns exactly max_new tokens: prompt token + 1, then + 1 per step
    for r in reqs:
        start = 100 * r.seq_id + 1
        assert r.generated == list(range(start, start + r.max_new)), (r.seq_id, r.generated)
    # step 0: requests 0 and 1 join; request 1 (2 tokens) is done after it.
    # step 1: 2 joins, 3 is done at its prefill (1 token), 4 joins: 3 rows.
    # steps 2-4: 2 and 4 run out; step 5 has nothing to run; 5 arrives at 6.
    assert [ids for ids, _ in e.launches] == [[0, 1], [0, 2, 4], [2, 4], [2, 4], [4], [5]]
    fin = {r.seq_id: r.finish_step for r in reqs}
    assert fin == {0: 1, 1: 0, 2: 3, 3: 1, 4: 4, 5: 6}
    assert out["finish_step"] == 6 and out["launches"] == 6 and out["steps"] == 7
    # released once each, right after the launch that gave the last token
    # (request 3, which needed no decode, after its prefill)
    assert dict(e.released) == {1: 1, 3: 1, 0: 2, 2: 4, 4: 5, 5: 6}
    assert not e.length


def test_a_full_batch_never_exceeds_max_batch():
    e = FakeEngine(max_batch=16)
    reqs = [_req(i, 4 + i, 3 + i % 5, i % 3) for i in range(40)]
    Batcher(e).run(reqs)
    assert max(len(ids) for ids, _ in e.launches) == 16
    assert all(len(r.generated) == r.max_new for r in reqs)
