"""Helpers shared by the GPU parity tests: run the CUDA path through the C
ABI binding, run the oracle on the same seeded inputs, compare."""
import numpy as np
import torch

import oracle
import image_preprocessing_gb300 as trfn

F32_TOL = 2e-6   # max-abs for binary32 output
F16_ULPS = 1     # binary16 output: at most one unit in the last place


def gpu_run(src, mean, std, aug=None, out_dtype=trfn.OUT_F32, layout=trfn.LAYOUT_NHWC,
            variant=trfn.VARIANT_AUTO, guard=0, src_offset=0, dst_offset=0, workspace=None):
    """Runs the CUDA kernel; returns the output as a numpy array (uint16 bits
    for binary16), and the guard bytes around it when guard > 0."""
    N, H, W, C = src.shape
    shape = trfn.out_shape(N, H, W, C, layout)
    ob = 2 if out_dtype == trfn.OUT_F16 else 4
    nbytes = int(np.prod(shape)) * ob
    dev = torch.device("cuda")
    s_buf = torch.empty(src.size + src_offset + 16, dtype=torch.uint8, device=dev)
    s_buf[src_offset:src_offset + src.size].copy_(torch.from_numpy(np.ascontiguousarray(src).reshape(-1)))
    d_buf = torch.full((nbytes + 2 * guard + dst_offset,), 0xAB, dtype=torch.uint8, device=dev)
    a = None
    if aug is not None:
        a = torch.from_numpy(np.ascontiguousarray(aug, dtype=np.int32)).to(dev)
    src_ptr = s_buf.data_ptr() + src_offset
    dst_ptr = d_buf.data_ptr() + guard + dst_offset
    trfn.tr_fused_norm(src_ptr, dst_ptr, mean, std, aug=a.data_ptr() if a is not None else None,
                       out_dtype=out_dtype, layout=layout, variant=variant, shape=(N, H, W, C),
                       workspace=workspace)
    torch.cuda.synchronize()
    host = d_buf.cpu().numpy()
    body = host[guard + dst_offset: guard + dst_offset + nbytes]
    out = body.view(np.uint16 if out_dtype == trfn.OUT_F16 else np.float32).reshape(shape)
    guards = np.concatenate([host[:guard + dst_offset], host[guard + dst_offset + nbytes:]])
    return out.copy(), guards


def f16_ulp_distance(a_bits, b_bits):
    """|a - b| in binary16 units in the last place (ordered integer view)."""
    def ordered(b):
        b = b.astype(np.int32)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(ordered(a_bits) - ordered(b_bits))


def assert_parity(gpu, ref, out_dtype, what=""):
    assert gpu.shape == ref.shape, what
    if out_dtype == trfn.OUT_F16:
        zero = ref == 0                     # +0 in the oracle (erased / padding)
        assert np.all(gpu[zero] == 0), "erased or padded elements are not +0 " + what
        d = f16_ulp_distance(gpu, ref)
        assert d.max(initial=0) <= F16_ULPS, "max fp16 ulp distance %d %s" % (d.max(), what)
    else:
        rb, gb = ref.view(np.uint32), gpu.view(np.uint32)
        assert np.all(gb[rb == 0] == 0), "erased or padded elements are not +0 " + what
        err = np.abs(gpu.astype(np.float64) - ref.astype(np.float64))
        assert err.max(initial=0) <= F32_TOL, "max abs error %g %s" % (err.max(), what)
        assert np.all(np.isfinite(gpu)), what


def zero_mask(out, layout, out_dtype):
    """Pixels whose every channel is exactly +0."""
    bits = out if out_dtype == trfn.OUT_F16 else out.view(np.uint32)
    if layout == trfn.LAYOUT_NCHW:
        return np.all(bits == 0, axis=1)
    if layout == trfn.LAYOUT_NHWC4:
        return np.all(bits[..., :3] == 0, axis=-1)
    return np.all(bits == 0, axis=-1)


def check_case(src, mean, std, aug, out_dtype, layout, variant=trfn.VARIANT_AUTO, guard=64, **kw):
    gpu, guards = gpu_run(src, mean, std, aug, out_dtype, layout, variant, guard=guard, **kw)
    ref = oracle.fused_norm(src, mean, std, aug, out_dtype=out_dtype, layout=layout)
    assert_parity(gpu, ref, out_dtype, "(shape %s dtype %d layout %d variant %d)" % (src.shape, out_dtype, layout, variant))
    assert np.all(guards == 0xAB), "bytes outside the output were written"
    return gpu, ref
