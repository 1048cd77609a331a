"""Host decode service (include/mk_service.h) on the CPU: the loop, the KV
page allocator, batching, park/resume, retiring -- driven by a Python step
function that records what the service hands the decode step.

"Cohere: a serving engine for North Mini Code built around a decode
megakernel", section "The inference engine around the kernel"."""
import numpy as np
import pytest

from moe_decode_megakernel_gb300 import MkError
from moe_decode_megakernel_gb300 import service as sv


class Recorder:
    """A step function: next token = (7 * token + seq_len) mod 1000; records
    every call and checks the block tables it is given."""

    def __init__(self, page_size, fail_at=None):
        self.P = page_size
        self.calls = []
        self.fail_at = fail_at

    def __call__(self, tok, sl, bt, out):
        if self.fail_at is not None and len(self.calls) == self.fail_at:
            self.fail_at = None
            return -2
        used = []
        for r in range(tok.size):
            n_pages = (sl[r] - 1) // self.P + 1  # pages covering positions 0 .. sl-1
            assert np.all(bt[r, :n_pages] >= 0), (sl[r], bt[r])
            assert np.all(bt[r, n_pages:] == -1), (sl[r], bt[r])
            used += bt[r, :n_pages].tolist()
        assert len(used) == len(set(used)), "two rows share a page"
        self.calls.append((tok.tolist(), sl.tolist(), bt.tolist()))
        out[:] = (7 * tok + sl) % 1000


def f(tok, sl):
    return (7 * tok + sl) % 1000


def test_prompt_then_samples():
    rec = Recorder(2)
    s = sv.Service(num_pages=8, page_size=2, max_pages=4, max_batch=2, step=rec)
    s.add(1, [5, 6, 7], max_new=3)
    out = s.run()
    # the prompt is fed one token per step; the output after the last prompt
    # token is the first sample, and each sample is fed at the next step
    t1 = f(7, 3)
    t2 = f(t1, 4)
    t3 = f(t2, 5)
    assert out == {1: [t1, t2, t3]}
    assert [c[0] for c in rec.calls] == [[5], [6], [7], [t1], [t2]]
    assert [c[1] for c in rec.calls] == [[1], [2], [3], [4], [5]]
    # a page per 2 positions, taken in increasing order
    assert rec.calls[-1][2] == [[0, 1, 2, -1]]
    info = s.query(1)
    assert info.state == sv.FINISHED and info.finish == sv.FIN_LENGTH and info.n_generated == 3
    assert s.free_pages == 8 and s.live == 0


def test_admission_order_and_batch_limit():
    rec = Recorder(4)
    s = sv.Service(num_pages=16, page_size=4, max_pages=4, max_batch=2, step=rec)
    for sid, tok in ((10, 100), (11, 200), (12, 300)):
        s.add(sid, [tok], max_new=2)
    rows, toks = s.step()
    assert rows == 2 and rec.calls[-1][0] == [100, 200]
    assert toks == [(10, f(100, 1)), (11, f(200, 1))]
    rows, toks = s.step()  # both finish (max_new 2)
    assert rows == 2 and [sid for sid, _ in toks] == [10, 11]
    rows, toks = s.step()  # now the third
    assert rows == 1 and rec.calls[-1][0] == [300] and toks == [(12, f(300, 1))]
    assert s.run() == {12: [f(f(300, 1), 2)]}


def test_park_keeps_pages_and_resume_feeds_appended_tokens():
    rec = Recorder(2)
    s = sv.Service(num_pages=8, page_size=2, max_pages=8, max_batch=4, step=rec)
    s.add(7, [1], max_new=4)
    _, a = s.step()
    _, b = s.step()
    t1, t2 = a[0][1], b[0][1]
    s.park(7)
    held = s.pages(7)
    assert s.step() == (0, []) and s.pages(7) == held and s.query(7).state == sv.PARKED
    s.resume(7, [900, 901])
    info = s.query(7)
    assert info.state == sv.RUNNING and info.n_pending == 3  # the last sample, then the two
    rows, toks = s.step()
    assert rec.calls[-1][0] == [t2] and toks == []  # fed, not a sample
    _, toks = s.step()
    assert rec.calls[-1][0] == [900] and toks == []
    _, toks = s.step()
    assert rec.calls[-1][0] == [901] and toks == [(7, f(901, 5))]
    out = s.run()
    assert out == {7: [f(f(901, 5), 6)]}
    assert s.query(7).finish == sv.FIN_LENGTH and s.query(7).n_ctx == 6
    del t1


def test_waits_for_a_free_page():
    rec = Recorder(2)
    s = sv.Service(num_pages=2, page_size=2, max_pages=4, max_batch=2, step=rec)
    s.add(1, [5, 6], max_new=1)  # positions 0, 1: one page
    s.add(2, [8, 9, 10], max_new=1)  # positions 0..2: two pages
    s.step()  # both take a page
    assert s.free_pages == 0
    rows, toks = s.step()  # seq 1 samples and retires; seq 2 feeds position 1
    assert rows == 2 and toks == [(1, f(6, 2))] and s.free_pages == 1
    rows, toks = s.step()  # seq 2 needs its second page: the one seq 1 gave back
    assert rows == 1 and toks == [(2, f(10, 3))]
    assert rec.calls[-1][2][0][:2] == [1, 0]
    assert s.free_pages == 2


def test_a_waiting_sequence_does_not_block_the_next():
    rec = Recorder(2)
    s = sv.Service(num_pages=1, page_size=2, max_pages=4, max_batch=2, step=rec)
    s.add(1, [1, 2, 3, 4], max_new=1)
    s.add(2, [5], max_new=1)
    s.step()  # seq 1 takes the only page
    rows, _ = s.step()  # seq 2 has no page: seq 1 runs alone
    assert rows == 1 and rec.calls[-1][0] == [2]
    rows, _ = s.step()  # seq 1 needs a second page: nobody can run
    assert rows == 0
    s.cancel(1)
    rows, toks = s.step()
    assert rows == 1 and toks == [(2, f(5, 1))]


def test_stop_token_and_context_limit():
    s = sv.Service(num_pages=8, page_size=2, max_pages=4, max_batch=2,
                   step=lambda tok, sl, bt, out: out.__setitem__(slice(None), 42))
    s.add(1, [3], max_new=10, stop_token=42)
    assert s.run() == {1: [42]} and s.query(1).finish == sv.FIN_STOP
    s2 = sv.Service(num_pages=8, page_size=2, max_pages=2, max_batch=2, step=Recorder(2))
    s2.add(1, [3, 4], max_new=10)
    out = s2.run()
    info = s2.query(1)
    assert info.finish == sv.FIN_CONTEXT and info.n_ctx == 4 and len(out[1]) == 3


def test_errors_and_forget():
    s = sv.Service(num_pages=4, page_size=2, max_pages=2, max_batch=1, step=Recorder(2))
    s.add(1, [3], max_new=2)
    with pytest.raises(MkError):
        s.add(1, [4], max_new=2)  # duplicate id
    with pytest.raises(MkError):
        s.add(2, [], max_new=2)
    with pytest.raises(MkError):
        s.resume(1)  # not parked
    with pytest.raises(MkError):
        s.park(99)
    with pytest.raises(MkError):
        s.forget(1)  # live
    s.step()
    s.cancel(1)
    assert s.query(1).finish == sv.FIN_CANCEL and s.free_pages == 4
    with pytest.raises(MkError):
        s.cancel(1)
    s.forget(1)
    s.add(1, [5], max_new=1)
    assert s.run() == {1: [f(5, 1)]}


def test_failed_step_changes_nothing():
    rec = Recorder(2, fail_at=2)
    s = sv.Service(num_pages=4, page_size=2, max_pages=4, max_batch=2, step=rec)
    s.add(1, [3, 4, 5], max_new=2)
    s.step()
    s.step()
    before = (s.query(1).n_ctx, s.query(1).n_pending, s.pages(1), s.free_pages)
    with pytest.raises(MkError):
        s.step()  # position 2 would take a page; the step fails
    assert (s.query(1).n_ctx, s.query(1).n_pending, s.pages(1), s.free_pages) == before
    out = s.run()  # the retry runs it
    assert out == {1: [f(5, 3), f(f(5, 3), 4)]}


def test_random_operations_keep_the_invariants():
    rng = np.random.default_rng(5)
    P, NP = 4, 24
    rec = Recorder(P)
    s = sv.Service(num_pages=NP, page_size=P, max_pages=6, max_batch=3, step=rec)
    live, next_id = set(), 0
    for _ in range(400):
        op = rng.integers(0, 10)
        if op < 2 and len(live) < 8:
            s.add(next_id, rng.integers(0, 1000, size=int(rng.integers(1, 9))), int(rng.integers(1, 12)))
            live.add(next_id)
            next_id += 1
        elif op == 2 and live:
            sid = int(rng.choice(sorted(live)))
            if s.query(sid).state == sv.RUNNING:
                s.park(sid)
            elif s.query(sid).state == sv.PARKED:
                s.resume(sid, rng.integers(0, 1000, size=int(rng.integers(0, 3))))
        elif op == 3 and live:
            sid = int(rng.choice(sorted(live)))
            if s.query(sid).state != sv.FINISHED:
                s.cancel(sid)
        else:
            s.step()
        held = []
        for sid in sorted(live):
            info = s.query(sid)
            pages = s.pages(sid)
            if info.state == sv.FINISHED:
                assert pages == []
                continue
            assert len(pages) == (info.n_ctx + P - 1) // P
            held += pages
        assert len(held) == len(set(held)) and len(held) + s.free_pages == NP
    for sid in sorted(live):
        if s.query(sid).state == sv.PARKED:
            s.resume(sid)
    s.run()
    assert s.live == 0 and s.free_pages == NP


def test_run_streams_tokens_in_order():
    rec = Recorder(4)
    s = sv.Service(num_pages=16, page_size=4, max_pages=4, max_batch=2, step=rec)
    s.add(1, [9, 8], max_new=3)
    s.add(2, [7], max_new=2)
    seen = []
    out = s.run(on_token=lambda sid, t: seen.append((sid, t)))
    assert [t for sid, t in seen if sid == 1] == out[1] and [t for sid, t in seen if sid == 2] == out[2]
    assert len(out[1]) == 3 and len(out[2]) == 2
    # step by step: 2 (prompt of 1) + 2 more for its samples ... all in 4 steps
    assert s.last_run_steps == 4 and len(rec.calls) == 4
    assert s.run(max_steps=5) == {} and s.last_run_steps == 0
