"""The host-side communicator's failure detection, without a GPU: virtual
ranks are host threads; count 0 makes a matched call a no-op, so only the
rendezvous, mismatch and timeout logic runs (the vasteelab page's hang
causes: a rank that never calls, differing count or type, a different call
order; and its advice to record each rank's last collective)."""
import threading
import time

import pytest
import torch

import gradient_allreduce_collective_gb300 as gar

F32, BF16 = torch.float32, torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def _lib():
    gar.build()
    gar.lib()


def _run(comm, calls):
    """calls[r] = kwargs for rank r (None: the rank never calls). Returns statuses."""
    out = [None] * len(calls)

    def go(r, kw):
        out[r] = comm.allreduce(r, 0x1000 * (r + 1), 0x100000 * (r + 1), **kw)

    ts = [threading.Thread(target=go, args=(r, kw)) for r, kw in enumerate(calls) if kw is not None]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=30)
    return out


def test_matching_calls_succeed_and_are_recorded():
    comm = gar.Comm(4, 2000)
    for k in range(2):
        st = _run(comm, [dict(count=0, dtype=F32, op="sum")] * 4)
        assert st == [0, 0, 0, 0]
    rec = comm.last_record(2)
    assert rec.seq == 2 and rec.status == 0 and rec.arrived_mask == 0b1111 and rec.count == 0


@pytest.mark.parametrize("bad", [dict(count=5, dtype=F32, op="sum"), dict(count=0, dtype=BF16, op="sum"),
                                 dict(count=0, dtype=F32, op="max")])
def test_mismatch_is_detected_before_launch_and_poisons(bad):
    comm = gar.Comm(4, 5000)
    good = dict(count=0, dtype=F32, op="sum")
    st = _run(comm, [good, good, bad, good])
    assert st == [gar.AR_ERR_MISMATCH] * 4
    masks = [comm.last_record(r).mismatch_mask for r in range(4)]
    assert any(m for m in masks)
    # the group is isolated: the next call fails at once with the same status
    t0 = time.perf_counter()
    assert _run(comm, [good] * 4) == [gar.AR_ERR_MISMATCH] * 4
    assert time.perf_counter() - t0 < 1.0


def test_missing_rank_times_out():
    comm = gar.Comm(4, 300)
    t0 = time.perf_counter()
    st = _run(comm, [dict(count=0, dtype=F32)] * 3 + [None])
    dt = time.perf_counter() - t0
    assert st[:3] == [gar.AR_ERR_TIMEOUT] * 3
    assert 0.25 < dt < 10
    rec = comm.last_record(0)
    assert rec.arrived_mask == 0b0111 and rec.status == gar.AR_ERR_TIMEOUT
    # the rank that finally calls finds the communicator poisoned
    assert comm.allreduce(3, 0x4000, 0x400000, count=0, dtype=F32) == gar.AR_ERR_TIMEOUT


def test_delayed_rank_within_timeout_records_skew():
    comm = gar.Comm(3, 5000)
    out = [None] * 3

    def go(r):
        if r == 2:
            time.sleep(0.15)
        out[r] = comm.allreduce(r, 0x1000, 0x100000 * (r + 1), count=0, dtype=F32)

    ts = [threading.Thread(target=go, args=(r,)) for r in range(3)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(timeout=30)
    assert out == [0, 0, 0]
    assert comm.last_record(2).arrival_skew_ms >= 100


def test_bad_arguments():
    with pytest.raises(gar.ArError):
        gar.Comm(0, 100)
    comm = gar.Comm(2, 100)
    assert comm.allreduce(5, 0x1000, 0x2000, count=0, dtype=F32) == gar.AR_ERR_INVALID_ARGUMENT
