"""Launches that overlap the kernel before them (tr_fused_norm_ex with
TR_LAUNCH_OVERLAP_PREVIOUS): consecutive batches with their own buffers and
workspaces alternating between two, eagerly and inside a CUDA graph, aligned
and odd-row forms, against the oracle; stream order for later work; the flag
dropped when a launch reuses the previous launch's workspace."""
import os

import numpy as np
import pytest

import oracle
import image_preprocessing_gb300 as trfn
from image_preprocessing_gb300 import synth
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

F16, F32 = trfn.OUT_F16, trfn.OUT_F32
NHWC, NCHW = trfn.LAYOUT_NHWC, trfn.LAYOUT_NCHW
MEAN = np.array(synth.IMAGENET_MEAN, np.float32)
STD = np.array(synth.IMAGENET_STD, np.float32)


def _bits(t, dt):
    import torch
    t = t.cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if dt == F16 else t.numpy()


def _batches(K, N, H, W, C, dt, layout, seed):
    import torch
    tdt = torch.float16 if dt == F16 else torch.float32
    srcs, recs, d_src, d_rec, dsts = [], [], [], [], []
    for k in range(K):
        src = synth.pixels_uniform(seed + k, N, H, W, C)
        rec, _ = oracle.sample_aug_params(seed + 100 + k, 0, N, H, W)
        srcs.append(src)
        recs.append(rec)
        d_src.append(torch.from_numpy(src).cuda())
        d_rec.append(torch.from_numpy(rec).cuda())
        dsts.append(torch.full(trfn.out_shape(N, H, W, C, layout), 7.0, dtype=tdt, device="cuda"))
    return srcs, recs, d_src, d_rec, dsts


def _check(srcs, recs, dsts, dt, layout):
    for k, (src, rec, dst) in enumerate(zip(srcs, recs, dsts)):
        ref = oracle.fused_norm(src, MEAN, STD, rec, out_dtype=dt, layout=layout)
        assert_parity(_bits(dst, dt), ref, dt, "overlapped batch %d" % k)


@pytest.mark.parametrize("shape,dt,layout,schedule", [
    ((64, 224, 224, 3), F16, NHWC, "dynamic"),
    ((64, 224, 224, 3), F32, NCHW, "static"),
    ((48, 299, 299, 3), F16, NHWC, "dynamic"),       # odd-row form
    ((256, 28, 28, 1), F32, NHWC, "dynamic"),        # odd-row form, small images
])
def test_consecutive_overlapped_launches(shape, dt, layout, schedule):
    import torch
    N, H, W, C = shape
    K = 6
    srcs, recs, d_src, d_rec, dsts = _batches(K, N, H, W, C, dt, layout, 4000 + W)
    wss = [torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda") for _ in range(2)]
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        for k in range(K):
            ws = wss[k % 2] if schedule == "dynamic" else None
            trfn.tr_fused_norm(d_src[k], dsts[k], MEAN, STD, d_rec[k], out_dtype=dt, layout=layout, stream=st,
                               workspace=ws, overlap_previous=True)
    torch.cuda.synchronize()
    _check(srcs, recs, dsts, dt, layout)
    for ws in wss:
        assert int(ws.count_nonzero()) == 0
    assert trfn.tr_device_status() == 0


def test_overlapped_launches_in_a_graph():
    import torch
    N, H, W, C = 64, 224, 224, 3
    K = 4
    srcs, recs, d_src, d_rec, dsts = _batches(K, N, H, W, C, F16, NHWC, 4500)
    wss = [torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda") for _ in range(2)]
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=st):
        for k in range(K):
            trfn.tr_fused_norm(d_src[k], dsts[k], MEAN, STD, d_rec[k], out_dtype=F16, stream=st,
                               workspace=wss[k % 2], overlap_previous=True)
    for rep in range(3):
        for d in dsts:
            d.fill_(5.0)
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            g.replay()
        torch.cuda.synchronize()
        _check(srcs, recs, dsts, F16, NHWC)
    for ws in wss:
        assert int(ws.count_nonzero()) == 0


def test_later_work_sees_both_launches():
    """A large launch, then a small overlapped one, then a torch copy of the
    large launch's output on the same stream: the copy sees it complete
    (the overlapped launch completes only after the one before it)."""
    import torch
    (src_a,), (rec_a,), (d_src_a,), (d_rec_a,), (dst_a,) = _batches(1, 256, 224, 224, 3, F16, NHWC, 4700)
    srcs_b, recs_b, d_src_b, d_rec_b, dsts_b = _batches(1, 8, 224, 224, 3, F16, NHWC, 4800)
    wss = [torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda") for _ in range(2)]
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    for rep in range(3):
        dst_a.fill_(3.0)
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            trfn.tr_fused_norm(d_src_a, dst_a, MEAN, STD, d_rec_a, out_dtype=F16, stream=st, workspace=wss[0])
            trfn.tr_fused_norm(d_src_b[0], dsts_b[0], MEAN, STD, d_rec_b[0], out_dtype=F16, stream=st,
                               workspace=wss[1], overlap_previous=True, variant=trfn.VARIANT_TILED)
            copy = dst_a.clone()
        torch.cuda.synchronize()
        ref = oracle.fused_norm(src_a, MEAN, STD, rec_a, out_dtype=F16)
        assert_parity(_bits(copy, F16), ref, F16, "copy after the overlapped launch")
    _check(srcs_b, recs_b, dsts_b, F16, NHWC)


def test_shared_workspace_drops_the_overlap():
    """The flag on launches that share one workspace: the library does not
    overlap them (their ticket counters would collide); results exact and the
    workspace zero again."""
    import torch
    N, H, W, C = 64, 224, 224, 3
    K = 5
    srcs, recs, d_src, d_rec, dsts = _batches(K, N, H, W, C, F16, NHWC, 4900)
    ws = torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda")
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        for k in range(K):
            trfn.tr_fused_norm(d_src[k], dsts[k], MEAN, STD, d_rec[k], out_dtype=F16, stream=st, workspace=ws,
                               overlap_previous=True)
    torch.cuda.synchronize()
    _check(srcs, recs, dsts, F16, NHWC)
    assert int(ws.count_nonzero()) == 0
    assert trfn.tr_device_status() == 0


def test_overlapped_crop_windows():
    """tr_fused_norm_crop_ex: consecutive crop launches overlapping, each with
    its own source, windows, records and output, workspaces alternating."""
    import torch
    N, H, W, C, S = 48, 224, 224, 3, 256
    K = 4
    wss = [torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda") for _ in range(2)]
    srcs, recs, crops, outs, d = [], [], [], [], []
    for k in range(K):
        src = synth.pixels_uniform(5100 + k, N, S, S, C)
        g = np.random.default_rng(5200 + k)
        crop = np.stack([g.integers(0, S - H + 1, N), g.integers(0, S - W + 1, N)], 1).astype(np.int32)
        rec, _ = oracle.sample_aug_params(5300 + k, 0, N, H, W)
        srcs.append(src); recs.append(rec); crops.append(crop)
        d.append((torch.from_numpy(src).cuda(), torch.from_numpy(crop).cuda(), torch.from_numpy(rec).cuda()))
        outs.append(torch.full((N, H, W, C), 7.0, dtype=torch.float16, device="cuda"))
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        for k in range(K):
            d_src, d_crop, d_rec = d[k]
            trfn.tr_fused_norm_crop(d_src, S, S, S * C, S * S * C, outs[k], N, H, W, C, MEAN, STD, crop=d_crop,
                                    aug=d_rec, out_dtype=F16, stream=st, workspace=wss[k % 2],
                                    overlap_previous=True)
    torch.cuda.synchronize()
    for k in range(K):
        win = np.stack([srcs[k][n, crops[k][n, 0]:crops[k][n, 0] + H, crops[k][n, 1]:crops[k][n, 1] + W]
                        for n in range(N)])
        ref = oracle.fused_norm(win, MEAN, STD, recs[k], out_dtype=F16)
        assert_parity(_bits(outs[k], F16), ref, F16, "overlapped crop batch %d" % k)
    for ws in wss:
        assert int(ws.count_nonzero()) == 0


def test_small_launches_never_run_ahead_of_a_large_one():
    """A large launch, then a chain of small overlapped launches alternating
    two workspaces, so launch k + 2 reuses launch k's workspace.  Small
    launches issue all their bands at once; were a launch to release its
    successor before its own predecessor completed, launch 2 could start
    while the large launch still holds the shared workspace's counters.  All
    outputs exact, workspaces zero, every time."""
    import torch
    (src_a,), (rec_a,), (d_src_a,), (d_rec_a,), (dst_a,) = _batches(1, 512, 224, 224, 3, F16, NHWC, 5500)
    K = 12
    srcs, recs, d_src, d_rec, dsts = _batches(K, 8, 224, 224, 3, F16, NHWC, 5600)
    wss = [torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda") for _ in range(2)]
    st = torch.cuda.Stream()
    ref_a = oracle.fused_norm(src_a, MEAN, STD, rec_a, out_dtype=F16)
    for rep in range(4):
        dst_a.fill_(3.0)
        for d in dsts:
            d.fill_(3.0)
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            trfn.tr_fused_norm(d_src_a, dst_a, MEAN, STD, d_rec_a, out_dtype=F16, stream=st, workspace=wss[0],
                               overlap_previous=True)
            for k in range(K):
                trfn.tr_fused_norm(d_src[k], dsts[k], MEAN, STD, d_rec[k], out_dtype=F16, stream=st,
                                   workspace=wss[(k + 1) % 2], overlap_previous=True, variant=trfn.VARIANT_TILED)
        torch.cuda.synchronize()
        assert_parity(_bits(dst_a, F16), ref_a, F16, "large launch, repetition %d" % rep)
        _check(srcs, recs, dsts, F16, NHWC)
        for ws in wss:
            assert int(ws.count_nonzero()) == 0
    assert trfn.tr_device_status() == 0


def test_random_overlapped_chains_match_waiting_launches():
    """About ten seconds (TRFN_CHAIN_SECONDS) of random chains of overlapped launches (sizes from
    2 to 512 images, aligned and odd-row forms, every layout, both types,
    host-made records and records drawn on the GPU in the same call,
    workspaces alternating, eager and replayed from graphs): every output and
    every GPU-made record equals, bit for bit, the same launch run without the
    option, and the workspaces are zero after every chain."""
    import time
    import torch
    rng = np.random.default_rng(11)
    shapes = [(256, 224, 224, 3), (8, 224, 224, 3), (64, 299, 299, 3), (512, 28, 28, 3), (2, 224, 224, 3),
              (128, 256, 256, 3), (16, 32, 32, 3), (96, 227, 227, 3)]
    bufs = []
    for i, (N, H, W, C) in enumerate(shapes):
        g = torch.Generator(device="cuda").manual_seed(300 + i)
        src = torch.randint(0, 256, (N, H, W, C), dtype=torch.uint8, device="cuda", generator=g)
        rec, _ = oracle.sample_aug_params(400 + i, 0, N, H, W)
        aug = torch.from_numpy(rec).cuda()
        dt = F16 if i % 2 == 0 else F32
        lay = (NHWC, NCHW, trfn.LAYOUT_NHWC4)[i % 3]
        tdt = torch.float16 if dt == F16 else torch.float32
        out = torch.empty(trfn.out_shape(N, H, W, C, lay), dtype=tdt, device="cuda")
        ref = torch.empty_like(out)
        sampled = i % 4 == 1
        rref = aug.clone()
        if sampled:
            trfn.tr_fused_norm_sampled(src, ref, MEAN, STD, 600 + i, 24 * i, rref, out_dtype=dt, layout=lay)
        else:
            trfn.tr_fused_norm(src, ref, MEAN, STD, aug, out_dtype=dt, layout=lay)
        bufs.append((src, aug, dt, lay, out, ref, sampled, i, rref))
    wss = [torch.zeros(trfn.tr_workspace_bytes(), dtype=torch.uint8, device="cuda") for _ in range(2)]
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    t0, chains = time.time(), 0
    seconds = float(os.environ.get("TRFN_CHAIN_SECONDS", "10"))   # longer stress runs set it
    while time.time() - t0 < seconds:
        order = rng.permutation(len(bufs)).tolist() + rng.integers(0, len(bufs), 4).tolist()
        seq = [order[0]] + [b for a, b in zip(order, order[1:]) if a != b]   # no buffer twice in a row

        def run():
            for k, j in enumerate(seq):
                src, aug, dt, lay, out, _, sampled, i, _ = bufs[j]
                if sampled:
                    trfn.tr_fused_norm_sampled(src, out, MEAN, STD, 600 + i, 24 * i, aug, out_dtype=dt, layout=lay,
                                               stream=st, workspace=wss[k % 2], overlap_previous=True)
                else:
                    trfn.tr_fused_norm(src, out, MEAN, STD, aug, out_dtype=dt, layout=lay, stream=st,
                                       workspace=wss[k % 2], overlap_previous=True)

        def reset():
            for b in bufs:
                b[4].fill_(7.0)
                if b[6]:
                    b[1].fill_(-9)
            torch.cuda.synchronize()
        reset()
        if chains % 3 == 2:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=st):
                run()
            reset()
            with torch.cuda.stream(st):
                graph.replay()
                graph.replay()
        else:
            with torch.cuda.stream(st):
                run()
        torch.cuda.synchronize()
        for j in set(seq):
            assert torch.equal(bufs[j][4], bufs[j][5]), "chain %d, buffer %d, sequence %s" % (chains, j, seq)
            assert torch.equal(bufs[j][1], bufs[j][8]), "records: chain %d, buffer %d" % (chains, j)
        for w in wss:
            assert int(w.count_nonzero()) == 0, "chain %d" % chains
        chains += 1
    assert chains > 100
    assert trfn.tr_device_status() == 0
