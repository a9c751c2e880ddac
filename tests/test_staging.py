"""Host staging zones (tr_stage_*): the producer side of the TransferStation.

Checks the hand-over the article "(10) Multi-threaded preprocessing, NUMA
awareness, asynchronous double buffering" (tech-renaissance.cn/blog/?p=481)
describes in §四 and §四.2, on the CPU with real threads (every ctypes call
releases the GIL): every sample lands in exactly one place, a batch turns
readable only when all its places are written, the last batch of closed data
is short, reproducible placement is independent of thread timing, and every
wait ends at its deadline.  No GPU: the staging area is pure host code.
"""
import threading
import time

import numpy as np
import pytest

import image_preprocessing_gb300 as trfn
from image_preprocessing_gb300 import Staging, TrError

H, W, C = 2, 3, 2           # 12-byte images: room for an 8-byte sample number
IMG = H * W * C


def zones(N):
    nb = trfn.tr_stage_zone_bytes(N, H, W, C)
    return [np.zeros(nb, np.uint8), np.zeros(nb, np.uint8)]


def write_sample(st, slot, value):
    img = st.image_view(slot)
    img.reshape(-1)[:8] = np.frombuffer(np.int64(value).tobytes(), np.uint8)
    img.reshape(-1)[8:] = value & 0xFF
    st.record_view(slot)[0, :] = (value & 1, value, -value, 0, 0)


def read_samples(st, b):
    imgs = st.image_view(b, b.count).reshape(b.count, -1)
    vals = imgs[:, :8].copy().view(np.int64).reshape(-1)
    assert np.array_equal(imgs[:, 8:], np.repeat((vals & 0xFF).astype(np.uint8)[:, None], IMG - 8, 1))
    recs = st.record_view(b, b.count)
    assert np.array_equal(recs[:, 1], vals) and np.array_equal(recs[:, 2], -vals)
    return vals


def consume_all(st, out, timeout_ms=20000):
    while True:
        b = st.wait_readable(timeout_ms)
        if b is None:
            return
        out.append((b.batch, b.count, read_samples(st, b)))
        st.release(b.batch)


def run_threads(targets):
    ts = [threading.Thread(target=t) for t in targets]
    for t in ts:
        t.start()
    return ts


def test_zone_bytes_layout():
    # [N images][pad to 256][N records of 20 bytes][pad to 256]
    assert trfn.tr_stage_zone_bytes(4, H, W, C) == 256 + 256
    assert trfn.tr_stage_zone_bytes(256, 224, 224, 3) == 38535168 + 5120
    assert trfn.tr_stage_zone_bytes(0, 1, 1, 1) == 0


@pytest.mark.parametrize("N,total,producers", [(8, 45, 6), (16, 2000, 8), (5, 25, 3), (7, 1, 2)])
def test_fast_mode_every_sample_once(N, total, producers):
    """Items from a shared source, places from the shared counter: each item
    in exactly one place, batches full except the last, in batch order."""
    st = Staging(zones(N), N, H, W, C, mode="fast")
    lock = threading.Lock()
    source = iter(range(total))
    errors = []

    def producer():
        try:
            while True:
                with lock:
                    item = next(source, None)
                if item is None:
                    return
                slot = st.acquire(timeout_ms=20000)
                assert slot is not None and slot.batch == slot.sample // N and slot.index == slot.sample % N
                write_sample(st, slot, item)
                st.commit(slot)
        except Exception as e:  # pragma: no cover - reported below
            errors.append(e)

    got = []
    consumer = threading.Thread(target=consume_all, args=(st, got))
    consumer.start()
    ps = run_threads([producer] * producers)
    for p in ps:
        p.join(60)
    assert not errors, errors
    st.close()           # every worker has run out: the samples handed out so far
    consumer.join(60)
    assert not consumer.is_alive()
    nb = (total + N - 1) // N
    assert [g[0] for g in got] == list(range(nb))
    assert [g[1] for g in got] == [N] * (total // N) + ([total % N] if total % N else [])
    items = np.concatenate([g[2] for g in got])
    assert sorted(items.tolist()) == list(range(total))
    assert st.acquire(timeout_ms=0) is None
    st.destroy()


def _reproducible_run(N, total, producers, delays_seed):
    st = Staging(zones(N), N, H, W, C, mode="reproducible")
    rng = np.random.default_rng(delays_seed)
    delays = rng.uniform(0, 2e-4, size=total)
    errors = []

    def producer(w):
        try:
            for s in range(w, total, producers):      # static assignment: worker w takes w, w+P, ...
                slot = st.acquire(s, timeout_ms=20000)
                assert slot.sample == s and slot.batch == s // N and slot.index == s % N
                time.sleep(delays[s])
                write_sample(st, slot, 1000003 * s % 999983)
                st.commit(slot)
        except Exception as e:  # pragma: no cover
            errors.append(e)

    got = []
    consumer = threading.Thread(target=consume_all, args=(st, got))
    consumer.start()
    ps = run_threads([(lambda w=w: producer(w)) for w in range(producers)])
    for p in ps:
        p.join(60)
    assert not errors, errors
    st.close(total)
    consumer.join(60)
    st.destroy()
    return got


def test_reproducible_mode_layout_independent_of_timing():
    N, total, P = 6, 40, 4
    a = _reproducible_run(N, total, P, 1)
    b = _reproducible_run(N, total, P, 2)
    expect = np.array([1000003 * s % 999983 for s in range(total)], np.int64)
    for run in (a, b):
        assert [g[0] for g in run] == list(range(7))
        assert [g[1] for g in run] == [6] * 6 + [4]
        assert np.array_equal(np.concatenate([g[2] for g in run]), expect)   # sample s at place s


def test_batch_readable_only_when_complete():
    N = 4
    st = Staging(zones(N), N, H, W, C, mode="reproducible")
    slots = [st.acquire(s, timeout_ms=0) for s in range(4)]
    for s in slots[:3]:
        write_sample(st, s, s.sample)
        st.commit(s)
    with pytest.raises(TrError) as e:
        st.wait_readable(timeout_ms=30)
    assert e.value.status == 4
    write_sample(st, slots[3], 3)
    st.commit(slots[3])
    b = st.wait_readable(timeout_ms=0)
    assert (b.batch, b.count) == (0, 4)
    assert read_samples(st, b).tolist() == [0, 1, 2, 3]
    st.release(0)
    st.destroy()


def test_acquire_waits_for_release_with_deadline():
    """Batch b + 2 shares batch b's zone: its producers wait until b is
    released, and give up at their deadline without claiming anything."""
    N = 2
    st = Staging(zones(N), N, H, W, C, mode="fast")
    for _ in range(4):                       # batches 0 and 1
        s = st.acquire(timeout_ms=0)
        write_sample(st, s, s.sample)
        st.commit(s)
    t0 = time.monotonic()
    with pytest.raises(TrError) as e:
        st.acquire(timeout_ms=60)            # batch 2: zone 0 still holds batch 0
    assert e.value.status == 4 and time.monotonic() - t0 >= 0.05
    b0 = st.wait_readable(timeout_ms=0)
    assert b0.batch == 0
    # a waiting producer is woken by the release
    got = {}

    def waiter():
        got["slot"] = st.acquire(timeout_ms=10000)

    t = threading.Thread(target=waiter)
    t.start()
    time.sleep(0.05)
    assert t.is_alive()
    st.release(0)
    t.join(10)
    assert got["slot"].sample == 4 and got["slot"].zone == 0   # the timed-out call claimed nothing
    b1 = st.wait_readable(timeout_ms=0)
    assert b1.batch == 1 and read_samples(st, b1).tolist() == [2, 3]
    st.destroy()


def test_close_short_last_batch_and_end():
    N = 4
    st = Staging(zones(N), N, H, W, C, mode="fast")
    slots = [st.acquire(timeout_ms=0) for _ in range(3)]
    st.close()                               # 3 handed out: one short batch
    assert st.acquire(timeout_ms=0) is None  # nothing handed out after the close
    with pytest.raises(TrError):
        st.wait_readable(timeout_ms=20)      # its places are not all written yet
    for s in slots:
        write_sample(st, s, 10 + s.sample)
        st.commit(s)
    b = st.wait_readable(timeout_ms=0)
    assert (b.batch, b.count) == (0, 3) and read_samples(st, b).tolist() == [10, 11, 12]
    st.release(0)
    assert st.wait_readable(timeout_ms=0) is None
    st.destroy()


def test_close_on_batch_boundary_and_empty():
    N = 3
    st = Staging(zones(N), N, H, W, C, mode="reproducible")
    for s in range(6):
        sl = st.acquire(s, timeout_ms=0)
        write_sample(st, sl, s)
        st.commit(sl)
    st.close(6)
    for k in range(2):
        b = st.wait_readable(timeout_ms=0)
        assert (b.batch, b.count) == (k, 3)
        st.release(k)
    assert st.wait_readable(timeout_ms=0) is None
    assert st.acquire(6, timeout_ms=0) is None
    st.destroy()
    st = Staging(zones(N), N, H, W, C)
    st.close()
    assert st.wait_readable(timeout_ms=0) is None
    st.destroy()


def test_argument_errors():
    N = 4
    z = zones(N)
    with pytest.raises(TrError):
        Staging([z[0], z[0]], N, H, W, C)                      # same zone twice
    with pytest.raises(TrError):
        Staging([z[0][:100], z[1][:100]], N, H, W, C)          # too small
    with pytest.raises(TrError):
        Staging(z, N, H, W, C, mode=7)
    st = Staging(z, N, H, W, C, mode="reproducible")
    with pytest.raises(TrError):
        st.acquire(-1, timeout_ms=0)
    s1 = st.acquire(1, timeout_ms=0)
    with pytest.raises(TrError):
        st.acquire(1, timeout_ms=0)                            # place already claimed
    st.commit(s1)
    with pytest.raises(TrError):
        st.commit(s1)                                          # committed twice
    with pytest.raises(TrError):
        st.release(0)                                          # not handed out
    with pytest.raises(TrError):
        st.close(1)                                            # sample 1 already claimed
    st.close(2)
    with pytest.raises(TrError):
        st.close(2)                                            # closed twice
    assert st.acquire(5, timeout_ms=0) is None                 # beyond the data
    s0 = st.acquire(0, timeout_ms=0)
    st.commit(s0)
    b = st.wait_readable(timeout_ms=0)
    assert (b.batch, b.count) == (0, 2)
    st.release(0)
    with pytest.raises(TrError):
        st.release(0)                                          # released twice
    with pytest.raises(TrError):
        st.acquire(0, timeout_ms=0)                            # batch 0 already consumed
    st.destroy()
    st = Staging(zones(N), N, H, W, C, mode="fast")
    st.acquire(timeout_ms=0)
    with pytest.raises(TrError):
        st.close(5)                                            # 1 handed out, not 5
    st.close(1)
    st.destroy()
