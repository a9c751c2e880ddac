"""Python face of libtrfn.so (the functions carry the C entry points' names).

PyTorch supplies device memory and streams only; each call below marshals
pointers, sizes and the stream handle into the C ABI declared in
include/tr_fused_norm.h and raises TrError on a non-zero status.
"""
import ctypes

import numpy as np

from . import _native
from ._native import AugParam, AugSampling, StageBatch, StageSlot, TrError, check, float_array, lib

OUT_F32, OUT_F16 = 0, 1
LAYOUT_NHWC, LAYOUT_NCHW, LAYOUT_NHWC4 = 0, 1, 2
VARIANT_AUTO, VARIANT_TILED, VARIANT_GENERIC = 0, 1, 2
LAUNCH_OVERLAP_PREVIOUS = 1   # tr_fused_norm_ex flags
PRESETS = {"NO_NORM": 0, "MNIST": 1, "CIFAR": 2, "IMAGENET": 3, "MLPERF": 4}

_DTYPES = {"f32": OUT_F32, "float32": OUT_F32, "f16": OUT_F16, "float16": OUT_F16}
_LAYOUTS = {"nhwc": LAYOUT_NHWC, "nchw": LAYOUT_NCHW, "nhwc4": LAYOUT_NHWC4}


def _code(v, table):
    return table[v.lower()] if isinstance(v, str) else int(v)


def out_shape(N, H, W, C, layout):
    layout = _code(layout, _LAYOUTS)
    if layout == LAYOUT_NCHW:
        return (N, C, H, W)
    if layout == LAYOUT_NHWC4:
        return (N, H, W, 4)
    return (N, H, W, C)


def _stream_handle(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev_ptr(t, what):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise TrError(1, what, "expects a CUDA tensor")
    if not t.is_contiguous():
        raise TrError(1, what, "expects a contiguous tensor")
    return t.data_ptr()


def _workspace_ptr(ws, where):
    """Device address of a scheduling workspace; a tensor must hold at least
    tr_workspace_bytes() bytes (the C ABI takes the pointer alone)."""
    if ws is None or isinstance(ws, int):
        return ws
    if ws.numel() * ws.element_size() < tr_workspace_bytes():
        raise TrError(1, where, "workspace must hold at least %d bytes" % tr_workspace_bytes())
    return _dev_ptr(ws, where)


def tr_fused_norm(src, dst, mean, std, aug=None, out_dtype=OUT_F16, layout=LAYOUT_NHWC, stream=None,
                  variant=VARIANT_AUTO, shape=None, workspace=None, overlap_previous=False):
    """Enqueue the fused step: src uint8 (N,H,W,C) CUDA tensor -> dst.

    dst: CUDA tensor of float32/float16 with out_shape(N,H,W,C,layout)
    elements; aug: CUDA int32 tensor (N,5) of {flip,y0,x0,h,w} or None;
    raw device addresses (ints) are accepted with shape=(N,H,W,C).
    workspace: zeroed CUDA buffer of tr_workspace_bytes() bytes for the
    dynamic band schedule (tr_fused_norm_ws), or None.
    overlap_previous: the caller's promise that this launch shares no buffer
    (workspace included) with the kernel before it in the stream
    (tr_fused_norm_ex with TR_LAUNCH_OVERLAP_PREVIOUS)."""
    dt = _code(out_dtype, _DTYPES)
    lay = _code(layout, _LAYOUTS)
    if shape is not None:
        N, H, W, C = shape
    else:
        import torch
        if src.dtype != torch.uint8 or src.dim() != 4:
            raise TrError(1, "tr_fused_norm", "src must be a uint8 (N,H,W,C) tensor")
        N, H, W, C = src.shape
        want = torch.float16 if dt == OUT_F16 else torch.float32
        if dst.dtype != want or dst.numel() != int(np.prod(out_shape(N, H, W, C, lay))):
            raise TrError(1, "tr_fused_norm", "dst must be %s with %d elements" % (want, np.prod(out_shape(N, H, W, C, lay))))
        if aug is not None and (aug.dtype != torch.int32 or aug.numel() != 5 * N):
            raise TrError(1, "tr_fused_norm", "aug must be int32 with N*5 elements")
    m, s = float_array(mean), float_array(std)
    rc = lib().tr_fused_norm_ex(_dev_ptr(src, "src"), _dev_ptr(dst, "dst"), N, H, W, C, m, s,
                                _dev_ptr(aug, "aug"), dt, lay, _stream_handle(stream), int(variant),
                                _workspace_ptr(workspace, "tr_fused_norm"),
                                LAUNCH_OVERLAP_PREVIOUS if overlap_previous else 0)
    check(rc, "tr_fused_norm")


def tr_fused_norm_batches(batches, mean, std, out_dtype=OUT_F16, layout=LAYOUT_NHWC, stream=None, shape=None,
                          workspace=None, overlap_previous=False):
    """The fused step on several batches of one shape in one launch.

    batches: list of (src, dst, aug) per batch -- CUDA tensors as for
    tr_fused_norm (aug may be None), or raw device addresses with
    shape=(N,H,W,C), the shape of ONE batch.  workspace and overlap_previous
    as tr_fused_norm."""
    dt = _code(out_dtype, _DTYPES)
    lay = _code(layout, _LAYOUTS)
    if shape is not None:
        N, H, W, C = shape
    else:
        import torch
        src0 = batches[0][0]
        if src0.dtype != torch.uint8 or src0.dim() != 4:
            raise TrError(1, "tr_fused_norm_batches", "sources must be uint8 (N,H,W,C) tensors")
        N, H, W, C = src0.shape
        want = torch.float16 if dt == OUT_F16 else torch.float32
        for src, dst, aug in batches:
            if tuple(src.shape) != (N, H, W, C) or src.dtype != torch.uint8:
                raise TrError(1, "tr_fused_norm_batches", "every source must be uint8 of one shape")
            if dst.dtype != want or dst.numel() != int(np.prod(out_shape(N, H, W, C, lay))):
                raise TrError(1, "tr_fused_norm_batches", "every dst must be %s of the output shape" % want)
            if aug is not None and (aug.dtype != torch.int32 or aug.numel() != 5 * N):
                raise TrError(1, "tr_fused_norm_batches", "aug must be int32 with N*5 elements")
    arr = (_native.Batch * max(1, len(batches)))()
    for k, (src, dst, aug) in enumerate(batches):
        arr[k] = _native.Batch(_dev_ptr(src, "src"), _dev_ptr(dst, "dst"), _dev_ptr(aug, "aug"))
    check(lib().tr_fused_norm_batches(arr, len(batches), N, H, W, C, float_array(mean), float_array(std), dt, lay,
                                      _stream_handle(stream), _workspace_ptr(workspace, "tr_fused_norm_batches"),
                                      LAUNCH_OVERLAP_PREVIOUS if overlap_previous else 0),
          "tr_fused_norm_batches")


def tr_fused_norm_sampled(src, dst, mean, std, seed, offset, records, flip=True, flip_p=0.5, erase=True,
                          erase_p=0.5, scale=(0.02, 0.33), ratio=(0.3, 3.3), out_dtype=OUT_F16, layout=LAYOUT_NHWC,
                          stream=None, variant=VARIANT_AUTO, workspace=None, overlap_previous=False):
    """tr_fused_norm with the records drawn on the GPU in the same launch
    (image n's record = tr_sample_aug_params_device's, counter block
    offset + 24n); records: CUDA int32 (N, 5) tensor receiving them;
    overlap_previous as tr_fused_norm (tr_fused_norm_sampled_ex).
    Returns the next free offset."""
    import torch
    if src.dtype != torch.uint8 or src.dim() != 4:
        raise TrError(1, "tr_fused_norm_sampled", "src must be a uint8 (N,H,W,C) tensor")
    N, H, W, C = src.shape
    dt, lay = _code(out_dtype, _DTYPES), _code(layout, _LAYOUTS)
    want = torch.float16 if dt == OUT_F16 else torch.float32
    if dst.dtype != want or dst.numel() != int(np.prod(out_shape(N, H, W, C, lay))):
        raise TrError(1, "tr_fused_norm_sampled", "dst must be %s of the output shape" % want)
    if records.dtype != torch.int32 or records.numel() != 5 * N:
        raise TrError(1, "tr_fused_norm_sampled", "records must be int32 with N*5 elements")
    sp = AugSampling(int(bool(flip)), float(flip_p), int(bool(erase)), float(erase_p), float(scale[0]),
                     float(scale[1]), float(ratio[0]), float(ratio[1]))
    nxt = ctypes.c_uint64(0)
    check(lib().tr_fused_norm_sampled_ex(_dev_ptr(src, "src"), _dev_ptr(dst, "dst"), N, H, W, C,
                                         float_array(mean), float_array(std), int(seed), int(offset),
                                         ctypes.byref(sp), _dev_ptr(records, "records"), ctypes.byref(nxt), dt, lay,
                                         _stream_handle(stream), int(variant),
                                         _workspace_ptr(workspace, "tr_fused_norm_sampled"),
                                         LAUNCH_OVERLAP_PREVIOUS if overlap_previous else 0),
          "tr_fused_norm_sampled")
    return nxt.value


def tr_fused_norm_crop(src, src_H, src_W, row_stride, image_stride, dst, N, H, W, C, mean, std, crop=None,
                       aug=None, out_dtype=OUT_F16, layout=LAYOUT_NHWC, stream=None, variant=VARIANT_AUTO,
                       workspace=None, overlap_previous=False):
    """Enqueue the fused step on H x W windows of a strided source.

    src: CUDA uint8 tensor (or device address) holding N images with the given
    row and image strides in bytes; crop: CUDA int32 (N, 2) {top, left} or
    None; dst: CUDA output with out_shape(N, H, W, C, layout) elements;
    overlap_previous as tr_fused_norm (tr_fused_norm_crop_ex)."""
    m, s = float_array(mean), float_array(std)
    rc = lib().tr_fused_norm_crop_ex(_dev_ptr(src, "src"), src_H, src_W, row_stride, image_stride,
                                     _dev_ptr(crop, "crop"), _dev_ptr(dst, "dst"), N, H, W, C, m, s,
                                     _dev_ptr(aug, "aug"), _code(out_dtype, _DTYPES), _code(layout, _LAYOUTS),
                                     _stream_handle(stream), int(variant),
                                     _workspace_ptr(workspace, "tr_fused_norm_crop"),
                                     LAUNCH_OVERLAP_PREVIOUS if overlap_previous else 0)
    check(rc, "tr_fused_norm_crop")


def tr_workspace_bytes():
    return int(lib().tr_workspace_bytes())


def tr_fused_norm_plan(src, dst, N, H, W, C, out_dtype, layout):
    v = ctypes.c_int(0)
    check(lib().tr_fused_norm_plan(src, dst, N, H, W, C, _code(out_dtype, _DTYPES), _code(layout, _LAYOUTS),
                                   ctypes.byref(v)), "tr_fused_norm_plan")
    return v.value


def tr_fused_norm_geometry(N, H, W, C, out_dtype=OUT_F16, layout=LAYOUT_NHWC, src=0x100000000, dst=0x200000000,
                           overlap_previous=False):
    """The TILED kernel's geometry for these arguments (tr_fused_norm_geometry):
    dict of rows, stages, ctas_per_sm, grid, odd_form.  src and dst are device
    addresses whose alignment the choice depends on (16-byte aligned
    defaults)."""
    out = [ctypes.c_int(0) for _ in range(5)]
    check(lib().tr_fused_norm_geometry(src, dst, N, H, W, C, _code(out_dtype, _DTYPES), _code(layout, _LAYOUTS),
                                       LAUNCH_OVERLAP_PREVIOUS if overlap_previous else 0,
                                       *[ctypes.byref(o) for o in out]), "tr_fused_norm_geometry")
    return dict(zip(("rows", "stages", "ctas_per_sm", "grid", "odd_form"), (o.value for o in out)))


def tr_norm_preset(preset):
    pid = PRESETS[preset] if isinstance(preset, str) else int(preset)
    m = (ctypes.c_float * 3)()
    s = (ctypes.c_float * 3)()
    ch = ctypes.c_int(0)
    check(lib().tr_norm_preset(pid, m, s, ctypes.byref(ch)), "tr_norm_preset")
    return (np.array(m[: ch.value], np.float32), np.array(s[: ch.value], np.float32), ch.value)


def tr_sample_aug_params(seed, offset, N, H, W, flip=True, flip_p=0.5, erase=True, erase_p=0.5,
                         scale=(0.02, 0.33), ratio=(0.3, 3.3)):
    """Host sampling of N records; returns (int32 array (N,5), next_offset)."""
    out = np.zeros((N, 5), np.int32)
    nxt = ctypes.c_uint64(0)
    check(lib().tr_sample_aug_params(seed, offset, N, H, W, int(bool(flip)), flip_p, int(bool(erase)), erase_p,
                                     scale[0], scale[1], ratio[0], ratio[1],
                                     out.ctypes.data_as(ctypes.c_void_p), ctypes.byref(nxt)),
          "tr_sample_aug_params")
    return out, nxt.value


def tr_sample_aug_params_device(seed, offset, N, H, W, out, flip=True, flip_p=0.5, erase=True, erase_p=0.5,
                                scale=(0.02, 0.33), ratio=(0.3, 3.3), stream=None):
    """Sample N records on the GPU into `out` (CUDA int32 (N, 5) tensor or a
    device address); returns the next offset (offset + 24 N)."""
    nxt = ctypes.c_uint64(0)
    check(lib().tr_sample_aug_params_device(seed, offset, N, H, W, int(bool(flip)), flip_p, int(bool(erase)),
                                            erase_p, scale[0], scale[1], ratio[0], ratio[1],
                                            _dev_ptr(out, "out"), ctypes.byref(nxt), _stream_handle(stream)),
          "tr_sample_aug_params_device")
    return nxt.value


def tr_validate_aug_params(records, H, W):
    """Returns -1 when every record is valid, else the first bad index."""
    rec = np.ascontiguousarray(records, dtype=np.int32).reshape(-1, 5)
    bad = ctypes.c_int(-1)
    rc = lib().tr_validate_aug_params(rec.ctypes.data_as(ctypes.c_void_p), rec.shape[0], H, W, ctypes.byref(bad))
    if rc not in (0, 1):
        check(rc, "tr_validate_aug_params")
    return bad.value


def tr_device_status(clear=False):
    v = ctypes.c_int(0)
    check(lib().tr_device_status(ctypes.byref(v), int(bool(clear))), "tr_device_status")
    return v.value


def tr_launch_count():
    return int(lib().tr_launch_count())


def tr_tune_tiled(band_bytes=0, stages=0, max_ctas_per_sm=0, flags=0):
    """Set the TILED kernel's geometry knobs (0 = default); see the C header."""
    check(lib().tr_tune_tiled(int(band_bytes), int(stages), int(max_ctas_per_sm), int(flags)), "tr_tune_tiled")


def tr_ts_slot_bytes(N, H, W, C):
    return int(lib().tr_ts_slot_bytes(N, H, W, C))


class TransferStation:
    """tr_ts_* wrapper: two caller-owned device input slots and three streams.

    The slots are CUDA uint8 tensors of tr_ts_slot_bytes(N,H,W,C) bytes each;
    the streams are torch.cuda.Stream objects (d2h may be None)."""

    def __init__(self, device, slots, copy_stream, compute_stream, d2h_stream=None):
        self._slots = slots  # keep the memory alive
        ptrs = (ctypes.c_void_p * 2)(slots[0].data_ptr(), slots[1].data_ptr())
        nbytes = min(slots[0].numel(), slots[1].numel())
        handle = ctypes.c_void_p(0)
        self.streams = (copy_stream, compute_stream, d2h_stream)
        check(lib().tr_ts_create(int(device), ptrs, nbytes, copy_stream.cuda_stream, compute_stream.cuda_stream,
                                 d2h_stream.cuda_stream if d2h_stream is not None else None,
                                 ctypes.byref(handle)), "tr_ts_create")
        self._h = handle

    def submit(self, h_src, d_dst, mean, std, h_params=None, h_dst=None, out_dtype=OUT_F16, layout=LAYOUT_NHWC):
        """h_src: pinned uint8 CPU tensor (N,H,W,C); d_dst: CUDA output tensor;
        h_params: pinned int32 CPU tensor (N,5) or None; h_dst: pinned CPU tensor or None."""
        N, H, W, C = h_src.shape
        k = ctypes.c_longlong(-1)
        check(lib().tr_ts_submit(self._h, h_src.data_ptr(), None if h_params is None else h_params.data_ptr(),
                                 d_dst.data_ptr(), None if h_dst is None else h_dst.data_ptr(), N, H, W, C,
                                 float_array(mean), float_array(std), _code(out_dtype, _DTYPES),
                                 _code(layout, _LAYOUTS), ctypes.byref(k)), "tr_ts_submit")
        return k.value

    def submit_partial(self, h_src, n_batch, d_dst, mean, std, h_params=None, h_dst=None, out_dtype=OUT_F16,
                       layout=LAYOUT_NHWC):
        """A short batch: h_src holds n_valid < n_batch images; the rest of the
        batch repeats the station's filler (first image of its first batch)."""
        n_valid, H, W, C = h_src.shape
        k = ctypes.c_longlong(-1)
        check(lib().tr_ts_submit_partial(self._h, h_src.data_ptr(),
                                         None if h_params is None else h_params.data_ptr(), n_valid,
                                         d_dst.data_ptr(), None if h_dst is None else h_dst.data_ptr(),
                                         n_batch, H, W, C, float_array(mean), float_array(std),
                                         _code(out_dtype, _DTYPES), _code(layout, _LAYOUTS), ctypes.byref(k)),
              "tr_ts_submit_partial")
        return k.value

    def submit_staged(self, staging, batch, d_dst, mean, std, n_batch=None, with_records=True, h_dst=None,
                      out_dtype=OUT_F16, layout=LAYOUT_NHWC):
        """Upload a batch handed out by staging.wait_readable() (a StageBatch),
        padded to n_batch images, run the kernel, and give the host zone back
        once its copies have finished."""
        N = staging.N if n_batch is None else n_batch
        _, H, W, C = staging.shape
        k = ctypes.c_longlong(-1)
        check(lib().tr_ts_submit_staged(self._h, staging._h, ctypes.byref(batch), int(bool(with_records)),
                                        d_dst.data_ptr(), None if h_dst is None else h_dst.data_ptr(), N, H, W, C,
                                        float_array(mean), float_array(std), _code(out_dtype, _DTYPES),
                                        _code(layout, _LAYOUTS), ctypes.byref(k)), "tr_ts_submit_staged")
        return k.value

    def sync(self, timeout_ms=-1):
        """True when all submitted work has finished; False on timeout."""
        rc = lib().tr_ts_sync(self._h, int(timeout_ms))
        if rc == 4:
            return False
        check(rc, "tr_ts_sync")
        return True

    def close(self):
        if self._h:
            h, self._h = self._h, None
            check(lib().tr_ts_destroy(h), "tr_ts_destroy")

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


STAGE_FAST, STAGE_REPRODUCIBLE = 0, 1
END_OF_DATA = 6
_STAGE_MODES = {"fast": STAGE_FAST, "reproducible": STAGE_REPRODUCIBLE}


def tr_stage_zone_bytes(N, H, W, C):
    return int(lib().tr_stage_zone_bytes(N, H, W, C))


class Staging:
    """tr_stage_* wrapper: two host zones that producer threads fill sample by
    sample while the station uploads the other zone.

    zones: two uint8 CPU tensors (pinned for asynchronous uploads) or numpy
    arrays of tr_stage_zone_bytes(N,H,W,C) bytes each.  acquire() returns a
    StageSlot (or None at the end of the data); image_view()/record_view()
    give numpy views of the slot's place."""

    def __init__(self, zones, N, H, W, C, mode=STAGE_FAST):
        self._zones = zones  # keep the memory alive
        ptrs = [z.data_ptr() if hasattr(z, "data_ptr") else z.ctypes.data for z in zones]
        nbytes = min(z.numel() if hasattr(z, "numel") else z.nbytes for z in zones)
        self._base = ptrs
        self.N, self.shape = N, (N, H, W, C)
        self.img_bytes = H * W * C
        handle = ctypes.c_void_p(0)
        check(lib().tr_stage_create((ctypes.c_void_p * 2)(*ptrs), nbytes, N, H, W, C,
                                    _code(mode, _STAGE_MODES), ctypes.byref(handle)), "tr_stage_create")
        self._h = handle

    def acquire(self, sample=-1, timeout_ms=-1):
        """A claimed StageSlot; None at the end of the data; raises TrError
        (status TR_ERR_TIMEOUT) when the deadline passes."""
        slot = StageSlot()
        rc = lib().tr_stage_acquire(self._h, int(sample), int(timeout_ms), ctypes.byref(slot))
        if rc == END_OF_DATA:
            return None
        check(rc, "tr_stage_acquire")
        return slot

    def commit(self, slot):
        check(lib().tr_stage_commit(self._h, ctypes.byref(slot)), "tr_stage_commit")

    def close(self, total_samples=-1):
        check(lib().tr_stage_close(self._h, int(total_samples)), "tr_stage_close")

    def wait_readable(self, timeout_ms=-1):
        """The next StageBatch in order; None after the last batch of closed data."""
        b = StageBatch()
        rc = lib().tr_stage_wait_readable(self._h, int(timeout_ms), ctypes.byref(b))
        if rc == END_OF_DATA:
            return None
        check(rc, "tr_stage_wait_readable")
        return b

    def release(self, batch):
        check(lib().tr_stage_release(self._h, int(batch)), "tr_stage_release")

    def _zone_offset(self, ptr, zone):
        return int(ptr) - int(self._base[zone])

    def image_view(self, slot_or_batch, count=1):
        """numpy uint8 view of `count` images starting at a slot's (or batch's) place."""
        zone = slot_or_batch.zone
        ptr = slot_or_batch.image if isinstance(slot_or_batch, StageSlot) else slot_or_batch.images
        z = self._zones[zone]
        arr = z.numpy() if hasattr(z, "numpy") else z
        off = self._zone_offset(ptr, zone)
        _, H, W, C = self.shape
        return arr[off:off + count * self.img_bytes].reshape(count, H, W, C)

    def record_view(self, slot_or_batch, count=1):
        """numpy int32 (count, 5) view of the records at a slot's (or batch's) place."""
        zone = slot_or_batch.zone
        ptr = slot_or_batch.record if isinstance(slot_or_batch, StageSlot) else slot_or_batch.records
        z = self._zones[zone]
        arr = z.numpy() if hasattr(z, "numpy") else z
        off = self._zone_offset(ptr, zone)
        return arr[off:off + count * 20].view(np.int32).reshape(count, 5)

    def destroy(self):
        if self._h:
            h, self._h = self._h, None
            check(lib().tr_stage_destroy(h), "tr_stage_destroy")

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.destroy()

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass
