"""Failure detection on the GPU without a fault: a pipeline wait that runs
out is reported through na3d_device_status, and the device stays usable.

na3d_selftest_withhold makes CTA 0 skip one of its K loads; the score
tile's wait for it gives up after ~2 s, the CTA drains its copies and MMAs,
frees its tensor memory and exits. Nothing faults or hangs."""
import ctypes

import numpy as np
import pytest
import torch

import na3d_inputs
import neighborhood_attention_video_gb300 as na
import oracle

pytestmark = pytest.mark.gpu


def to_dev(a):
    return torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("shape,kernel", [
    ((1, 4, 8, 16, 2, 32), (3, 5, 5)),     # W window by the tensor core
    ((1, 4, 8, 5, 2, 64), (3, 5, 5)),      # whole-row W windows: H window by the tensor core
    ((1, 5, 9, 40, 2, 64), (3, 5, 33)),    # per-key masks
    ((1, 6, 12, 16, 3, 64), (3, 1, 3)),    # HD 64, 96-key score tiles in pairs of slots
    ((1, 2, 4, 6, 1, 512), (1, 3, 5)),     # HD 512: Q and K streamed per region
], ids=lambda x: "x".join(map(str, x)))
def test_withheld_load_is_reported_and_the_device_stays_usable(shape, kernel):
    q, k, v = na3d_inputs.make_qkv(*shape, seed=41)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    out = torch.empty_like(qd)
    lib = na.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    assert na.na3d_device_status() == 0
    P = ctypes.c_void_p
    rc = lib.na3d_selftest_withhold(P(qd.data_ptr()), P(kd.data_ptr()), P(vd.data_ptr()),
                                    P(out.data_ptr()), *shape, *kernel, 1, P(stream))
    assert rc == 0
    assert na.na3d_device_status() == 10          # NA3D_ERR_DEVICE_TIMEOUT, flag cleared
    assert na.na3d_device_status() == 0
    # the same context computes correctly afterwards
    out2 = torch.empty_like(qd)
    na.na3d_fwd(qd, kd, vd, out2, kernel)
    torch.cuda.synchronize()
    assert na.na3d_device_status() == 0
    got = na3d_inputs.bf16_bits_to_f64(out2.view(torch.int16).cpu().numpy().view(np.uint16))
    want = oracle.na3d_fwd(q, k, v, kernel)
    assert float(np.linalg.norm(got - want) / np.linalg.norm(want)) <= 5e-3


def test_a_timeout_is_taken_by_exactly_one_status_call():
    """Two status calls on two streams from two host threads, after one
    timed-out launch: the flag is read and cleared in one atomic step, so
    exactly one call reports it."""
    import threading
    shape, kernel = (1, 4, 8, 16, 2, 32), (3, 5, 5)
    q, k, v = na3d_inputs.make_qkv(*shape, seed=43)
    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    out = torch.empty_like(qd)
    lib = na.load_library()
    assert na.na3d_device_status() == 0
    P = ctypes.c_void_p
    rc = lib.na3d_selftest_withhold(P(qd.data_ptr()), P(kd.data_ptr()), P(vd.data_ptr()),
                                    P(out.data_ptr()), *shape, *kernel, 0,
                                    P(torch.cuda.current_stream().cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    results = [None, None]
    go = threading.Barrier(2)

    def take(i):
        torch.cuda.set_device(0)
        go.wait()
        results[i] = na.na3d_device_status(streams[i])

    threads = [threading.Thread(target=take, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert sorted(results) == [0, 10], results
    assert na.na3d_device_status() == 0
