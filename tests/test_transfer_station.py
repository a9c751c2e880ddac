"""The transfer station (double-buffered feeding from pinned host memory):
every batch's output equals the direct kernel's, slots are reused only after
the kernel that read them, results come back to pinned host buffers, and
tr_ts_sync gives up at its deadline without losing the queued work.

The A/B hand-over follows the TransferStation of the Tech-Renaissance article
"(10) Multi-threaded preprocessing, NUMA awareness, asynchronous double
buffering" (tech-renaissance.cn/blog/?p=481, §四)."""
import numpy as np
import pytest

import oracle
import image_preprocessing_gb300 as trfn
from image_preprocessing_gb300 import synth
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

MEAN = np.array(synth.IMAGENET_MEAN, np.float32)
STD = np.array(synth.IMAGENET_STD, np.float32)


def _station(N, H, W, C, with_d2h=True):
    import torch
    nbytes = trfn.tr_ts_slot_bytes(N, H, W, C)
    slots = [torch.empty(nbytes, dtype=torch.uint8, device="cuda") for _ in range(2)]
    streams = [torch.cuda.Stream() for _ in range(3)]
    ts = trfn.TransferStation(torch.cuda.current_device(), slots, streams[0], streams[1],
                              streams[2] if with_d2h else None)
    return ts, streams


@pytest.mark.parametrize("dt", [trfn.OUT_F16, trfn.OUT_F32])
def test_every_batch_matches_the_oracle(dt):
    import torch
    N, H, W, C = 8, 32, 48, 3
    K = 7
    ts, _ = _station(N, H, W, C)
    tdt = torch.float16 if dt == trfn.OUT_F16 else torch.float32
    srcs = [synth.pixels_gaussian(300 + k, N, H, W, C) for k in range(K)]
    recs = [oracle.sample_aug_params(400 + k, 0, N, H, W)[0] for k in range(K)]
    h_src = [torch.from_numpy(x).pin_memory() for x in srcs]
    h_par = [torch.from_numpy(r).pin_memory() for r in recs]
    d_out = [torch.empty((N, H, W, C), dtype=tdt, device="cuda") for _ in range(K)]
    h_out = [torch.zeros((N, H, W, C), dtype=tdt).pin_memory() for _ in range(K)]
    for k in range(K):
        assert ts.submit(h_src[k], d_out[k], MEAN, STD, h_params=h_par[k], h_dst=h_out[k], out_dtype=dt) == k
    assert ts.sync(30000)
    for k in range(K):
        ref = oracle.fused_norm(srcs[k], MEAN, STD, recs[k], out_dtype=dt)
        for got in (d_out[k].cpu(), h_out[k]):
            arr = got.view(torch.int16).numpy().view(np.uint16) if dt == trfn.OUT_F16 else got.numpy()
            assert_parity(arr, ref, dt, "batch %d" % k)
    ts.close()


def test_two_device_outputs_reused_across_batches():
    """d_dst alternating between two buffers while results are copied back:
    batch k's kernel waits for batch k-2's copy to the host."""
    import torch
    N, H, W, C = 4, 16, 32, 3
    K = 9
    ts, _ = _station(N, H, W, C)
    srcs = [synth.pixels_uniform(500 + k, N, H, W, C) for k in range(K)]
    h_src = [torch.from_numpy(x).pin_memory() for x in srcs]
    d_out = [torch.empty((N, H, W, C), dtype=torch.float16, device="cuda") for _ in range(2)]
    h_out = [torch.zeros((N, H, W, C), dtype=torch.float16).pin_memory() for _ in range(K)]
    for k in range(K):
        ts.submit(h_src[k], d_out[k % 2], MEAN, STD, h_dst=h_out[k])
    assert ts.sync(30000)
    for k in range(K):
        ref = oracle.fused_norm(srcs[k], MEAN, STD, None, out_dtype=trfn.OUT_F16)
        assert_parity(h_out[k].view(torch.int16).numpy().view(np.uint16), ref, trfn.OUT_F16, "batch %d" % k)
    ts.close()


def test_sync_times_out_then_completes():
    """A copy stream held busy by a bounded sleep kernel: a short sync gives up
    with a timeout, a later unbounded sync sees the batch complete."""
    import torch
    N, H, W, C = 2, 8, 16, 3
    ts, (s_copy, s_comp, s_d2h) = _station(N, H, W, C)
    src = synth.pixels_uniform(7, N, H, W, C)
    h_src = torch.from_numpy(src).pin_memory()
    d_out = torch.empty((N, H, W, C), dtype=torch.float16, device="cuda")
    with torch.cuda.stream(s_copy):
        torch.cuda._sleep(400_000_000)   # a few hundred milliseconds of spinning, bounded
    ts.submit(h_src, d_out, MEAN, STD)
    assert ts.sync(5) is False
    assert ts.sync(-1) is True
    ref = oracle.fused_norm(src, MEAN, STD, None, out_dtype=trfn.OUT_F16)
    assert_parity(d_out.cpu().view(torch.int16).numpy().view(np.uint16), ref, trfn.OUT_F16)
    ts.close()


def test_submit_rejects_bad_arguments():
    import torch
    N, H, W, C = 2, 8, 16, 3
    ts, _ = _station(N, H, W, C, with_d2h=False)
    h_src = torch.zeros((N, H, W, C), dtype=torch.uint8).pin_memory()
    d_out = torch.empty((N, H, W, C), dtype=torch.float16, device="cuda")
    h_out = torch.zeros((N, H, W, C), dtype=torch.float16).pin_memory()
    with pytest.raises(trfn.TrError):
        ts.submit(h_src, d_out, MEAN, STD, h_dst=h_out)   # no result stream was given
    big = torch.zeros((10 * N, H, W, C), dtype=torch.uint8).pin_memory()
    assert 10 * N * H * W * C > trfn.tr_ts_slot_bytes(N, H, W, C)
    with pytest.raises(trfn.TrError):
        ts.submit(big, d_out, MEAN, STD)                   # does not fit a slot
    ts.close()


def _f16(t):
    import torch
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def test_short_batch_is_padded_with_the_first_batchs_first_image():
    """TransferStation §四.1: a short last batch is filled up with the first
    sample of the first batch, so every batch keeps one size."""
    import torch
    N, H, W, C = 6, 16, 32, 3
    ts, _ = _station(N, H, W, C)
    full = synth.pixels_uniform(61, N, H, W, C)
    short = synth.pixels_uniform(62, 2, H, W, C)
    r_full = oracle.sample_aug_params(63, 0, N, H, W)[0]
    r_short = oracle.sample_aug_params(64, 0, 2, H, W)[0]
    d0 = torch.empty((N, H, W, C), dtype=torch.float16, device="cuda")
    d1 = torch.empty((N, H, W, C), dtype=torch.float16, device="cuda")
    ts.submit(torch.from_numpy(full).pin_memory(), d0, MEAN, STD, h_params=torch.from_numpy(r_full).pin_memory())
    ts.submit_partial(torch.from_numpy(short).pin_memory(), N, d1, MEAN, STD,
                      h_params=torch.from_numpy(r_short).pin_memory())
    assert ts.sync(30000)
    want_src = np.concatenate([short, np.repeat(full[:1], N - 2, axis=0)])
    want_rec = np.concatenate([r_short, np.repeat(r_full[:1], N - 2, axis=0)])
    ref = oracle.fused_norm(want_src, MEAN, STD, want_rec, out_dtype=trfn.OUT_F16)
    assert_parity(_f16(d1), ref, trfn.OUT_F16, "padded batch")
    ref0 = oracle.fused_norm(full, MEAN, STD, r_full, out_dtype=trfn.OUT_F16)
    assert_parity(_f16(d0), ref0, trfn.OUT_F16, "first batch")
    ts.close()


def test_first_batch_short_pads_with_its_own_first_image():
    import torch
    N, H, W, C = 4, 8, 16, 3
    ts, _ = _station(N, H, W, C)
    short = synth.pixels_uniform(71, 1, H, W, C)
    d = torch.empty((N, H, W, C), dtype=torch.float16, device="cuda")
    ts.submit_partial(torch.from_numpy(short).pin_memory(), N, d, MEAN, STD)
    assert ts.sync(30000)
    ref = oracle.fused_norm(np.repeat(short, N, axis=0), MEAN, STD, None, out_dtype=trfn.OUT_F16)
    assert_parity(_f16(d), ref, trfn.OUT_F16)
    with pytest.raises(trfn.TrError):
        ts.submit_partial(torch.from_numpy(np.repeat(short, N + 1, axis=0)).pin_memory(), N, d, MEAN, STD)
    ts.close()


def _staged_pipeline(mode, N, H, W, C, T, producers, dt=trfn.OUT_F16):
    """Producer threads write samples into pinned host zones (tr_stage_*); the
    consumer submits each readable batch to the station, which gives the zone
    back once its upload has finished.  Returns per batch (place -> sample,
    count, device output)."""
    import threading
    import torch
    data = synth.pixels_uniform(900, T, H, W, C)
    recs = oracle.sample_aug_params(901, 0, T, H, W)[0]
    nb = trfn.tr_stage_zone_bytes(N, H, W, C)
    zones = [torch.zeros(nb, dtype=torch.uint8).pin_memory() for _ in range(2)]
    st = trfn.Staging(zones, N, H, W, C, mode=mode)
    ts, _ = _station(N, H, W, C)
    lock = threading.Lock()
    source = iter(range(T))
    placed = {}            # sample number (place) -> data item
    errors = []

    def producer(w):
        try:
            mine = iter(range(w, T, producers))
            while True:
                if mode == trfn.STAGE_FAST:
                    with lock:
                        item = next(source, None)
                    if item is None:
                        return
                    slot = st.acquire(timeout_ms=30000)
                else:
                    item = next(mine, None)
                    if item is None:
                        return
                    slot = st.acquire(item, timeout_ms=30000)
                st.image_view(slot)[0] = data[item]
                st.record_view(slot)[0] = recs[item]
                with lock:
                    placed[slot.sample] = item
                st.commit(slot)
        except Exception as e:  # pragma: no cover
            errors.append(e)

    threads = [threading.Thread(target=producer, args=(w,)) for w in range(producers)]
    for t in threads:
        t.start()
    tdt = torch.float16 if dt == trfn.OUT_F16 else torch.float32
    outs = []
    closed = False
    while True:
        if not closed and not any(t.is_alive() for t in threads):
            st.close()
            closed = True
        try:
            b = st.wait_readable(timeout_ms=50)
        except trfn.TrError as e:
            assert e.status == 4
            continue
        if b is None:
            break
        d = torch.empty((N, H, W, C), dtype=tdt, device="cuda")
        assert ts.submit_staged(st, b, d, MEAN, STD, out_dtype=dt) == b.batch
        outs.append((b.batch, b.count, d))
    assert ts.sync(30000)
    for t in threads:
        t.join(10)
    assert not errors, errors
    ts.close()
    st.destroy()
    return data, recs, placed, outs


@pytest.mark.parametrize("mode", [0, 1])
def test_staged_batches_match_the_oracle(mode):
    """Every place of every batch, including the short last batch's filler
    images (the first image and record of the first batch), equals the
    oracle on the sample the producers put there."""
    N, H, W, C = 8, 32, 48, 3
    T = 5 * N + 3
    data, recs, placed, outs = _staged_pipeline(mode, N, H, W, C, T, producers=4)
    assert [o[0] for o in outs] == list(range(6))
    assert [o[1] for o in outs] == [N] * 5 + [3]
    assert sorted(placed) == list(range(T)) and sorted(placed.values()) == list(range(T))
    if mode == 1:
        assert all(placed[s] == s for s in placed)             # reproducible: sample s at place s
    filler = placed[0]
    for b, count, d in outs:
        items = [placed[b * N + i] if i < count else filler for i in range(N)]
        ref = oracle.fused_norm(data[items], MEAN, STD, recs[items], out_dtype=trfn.OUT_F16)
        got = d.cpu().view(__import__("torch").int16).numpy().view(np.uint16)
        assert_parity(got, ref, trfn.OUT_F16, "staged batch %d" % b)


def test_full_size_stream_with_a_short_last_batch_matches_the_oracle():
    """The stream workload at full size (TransferStation §四, §四.1): four
    256 x 224x224x3 batches of clipped-Gaussian pixels with flip and erase
    records (Philox offsets running on across batches) go through
    tr_ts_submit, then a short batch of 100 images through
    tr_ts_submit_partial, which pads it with the first batch's first image and
    record.  Every element of every batch, on the device and copied back to
    pinned host memory, against the oracle."""
    import concurrent.futures as cf
    import torch
    N, H, W, C = 256, 224, 224, 3
    B, short = 4, 100
    ts, _ = _station(N, H, W, C)
    h_src = [torch.empty((N if b < B else short, H, W, C), dtype=torch.uint8).pin_memory() for b in range(B + 1)]
    for b in range(B + 1):
        synth.pixels_gaussian_into(5000 + b, h_src[b].numpy())
    recs, offset = [], 0
    for b in range(B + 1):
        r, offset = oracle.sample_aug_params(2005, offset, h_src[b].shape[0], H, W)
        recs.append(r)
    h_par = [torch.from_numpy(r).pin_memory() for r in recs]
    d_out = [torch.empty((N, H, W, C), dtype=torch.float16, device="cuda") for _ in range(B + 1)]
    h_out = [torch.zeros((N, H, W, C), dtype=torch.float16).pin_memory() for _ in range(B + 1)]
    for b in range(B):
        assert ts.submit(h_src[b], d_out[b], MEAN, STD, h_params=h_par[b], h_dst=h_out[b]) == b
    assert ts.submit_partial(h_src[B], N, d_out[B], MEAN, STD, h_params=h_par[B], h_dst=h_out[B]) == B
    assert ts.sync(60000)
    ts.close()
    first_img, first_rec = h_src[0].numpy()[:1], recs[0][:1]
    srcs = [h_src[b].numpy() for b in range(B)] + [
        np.concatenate([h_src[B].numpy(), np.repeat(first_img, N - short, axis=0)])]
    rs = recs[:B] + [np.concatenate([recs[B], np.repeat(first_rec, N - short, axis=0)])]

    def reference(b, lo, hi):
        return oracle.fused_norm(srcs[b][lo:hi], MEAN, STD, rs[b][lo:hi], out_dtype=trfn.OUT_F16)

    step = 16
    with cf.ThreadPoolExecutor(max_workers=8) as ex:
        for b in range(B + 1):
            ref = np.concatenate(list(ex.map(lambda lo: reference(b, lo, lo + step), range(0, N, step))))
            assert_parity(_f16(d_out[b]), ref, trfn.OUT_F16, "device output of batch %d" % b)
            assert_parity(h_out[b].view(torch.int16).numpy().view(np.uint16), ref, trfn.OUT_F16,
                          "host copy of batch %d" % b)
