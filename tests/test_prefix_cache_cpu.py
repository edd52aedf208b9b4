"""Prefix reuse on the page pool, host side (no GPU): `engine.PrefixCache`
over a fake engine that records the calls the cache makes.  The workload is
the one "rec Megakernel and Tempo9 Compared", §1 (Prefix cache) describes: a
second turn over the same 8,022-token prompt reuses 7,936 of its tokens (62
whole 128-token pages), a different prompt reuses nothing, and returning to
the first prompt reuses it again while its entry is held."""
import torch

from moe_decode_megakernel_persistent_gb300.engine import PrefixCache


class FakeEngine:
    def __init__(self):
        self.calls = []

    def fork(self, src, dst, n_tokens):
        self.calls.append(("fork", src, dst, n_tokens))

    def prefill(self, seq_id, tokens, start_pos=0, out=None):
        self.calls.append(("prefill", seq_id, start_pos, int(tokens.numel())))
        return "next-token"

    def release(self, seq_id):
        self.calls.append(("release", seq_id))


def _prompt(seed, n):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, 151936, (n,), generator=g, dtype=torch.int32)


def test_a_a_b_a_turns_reuse_whole_pages():
    e = FakeEngine()
    pc = PrefixCache(e, capacity=4)
    a = _prompt(1, 8022)
    # turn 1: nothing cached, the whole prompt is prefilled
    out, n = pc.prefill(0, a)
    assert (out, n) == ("next-token", 0) and e.calls == [("prefill", 0, 0, 8022)]
    pc.keep(0, a.tolist())
    # turn 2: the same prompt plus 40 new tokens shares 62 pages = 7,936 tokens
    e.calls.clear()
    a2 = torch.cat([a, _prompt(2, 40)])
    _, n = pc.prefill(1, a2)
    assert n == 7936 == 62 * 128
    assert e.calls == [("fork", 0, 1, 7936), ("prefill", 1, 7936, 8062 - 7936)]
    pc.keep(1, a2.tolist())
    # turn 3: a different prompt shares nothing
    e.calls.clear()
    b = _prompt(3, 5000)
    _, n = pc.prefill(2, b)
    assert n == 0 and e.calls == [("prefill", 2, 0, 5000)]
    pc.keep(2, b.tolist())
    # turn 4: back to the first prompt; the longest held match is turn 2's entry
    e.calls.clear()
    _, n = pc.prefill(3, a)
    assert n == 7936 and e.calls[0][0] == "fork" and e.calls[0][3] == 7936
    assert e.calls[1] == ("prefill", 3, 7936, 8022 - 7936)


def test_at_least_one_token_is_prefilled_and_short_prompts_share_nothing():
    e = FakeEngine()
    pc = PrefixCache(e)
    p = _prompt(4, 256)                    # exactly two pages
    pc.prefill(0, p)
    pc.keep(0, p.tolist())
    e.calls.clear()
    _, n = pc.prefill(1, p)                # the same 256 tokens: the last must be prefilled
    assert n == 128 and e.calls[-1] == ("prefill", 1, 128, 128)
    e.calls.clear()
    _, n = pc.prefill(2, p[:100])          # shorter than a page
    assert n == 0 and e.calls == [("prefill", 2, 0, 100)]


def test_longest_match_wins_and_least_recently_used_is_evicted():
    e = FakeEngine()
    pc = PrefixCache(e, capacity=2)
    base = _prompt(5, 1000)
    short = torch.cat([base[:300], _prompt(6, 200)])   # shares 2 pages with base
    pc.keep(10, short.tolist())
    pc.keep(11, base.tolist())
    _, n = pc.prefill(12, torch.cat([base, _prompt(7, 10)]))
    assert n == 896 and e.calls[0] == ("fork", 11, 12, 896)   # 7 pages of base, not short's 2
    # the entry just used moved to the back: keeping a third evicts `short`
    pc.keep(13, _prompt(8, 50).tolist())
    assert ("release", 10) in e.calls and ("release", 11) not in e.calls
    assert [sid for sid, _ in pc.entries] == [11, 13]
