"""The allocation-free GEMV entry point, checked against tf_gemv.

tf_gemv_noalloc exists for callers that cannot allocate device memory where
they run a layer (inside another framework's memory pool, in a plugin that
only receives input and output pointers, on a latency-critical path where an
allocation may block or fail).  Its split-K scratch is a fixed array inside
libtf instead of a caller-provided workspace.  This test calls it through the
C ABI, twice in a row on the same stream (so the second call runs on the
scratch the first one left behind), and compares each result with the
existing tf_gemv entry point within the parity tolerance of the other tests.

The file is named to be collected last, so that a run stopping at the first
failure has run every other test before this one.
"""

import ctypes

import numpy as np
import pytest

import gemv_tf_prepack_gb300 as tf
from gemv_tf_prepack_gb300 import synth
from oracle import tf_oracle
from tests._gpu_util import check_close, layer, to_dev_bf16, to_host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gemv_tf_prepack_gb300 import build as b
    b.build()
    import torch
    torch.cuda.set_device(0)
    yield
    assert tf.device_error() == 0


def _noalloc(W, x, y):
    import torch
    rc = tf.lib().tf_gemv_noalloc(ctypes.c_void_p(W.blob.data_ptr()), W.nbytes, W.N, W.K, W.bits, W.group,
                                  ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(y.data_ptr()), x.shape[0],
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, tf.lib().tf_status_string(rc).decode()
    return y


@pytest.mark.parametrize("N,K,bits,group,M", [
    (4096, 4096, 4, 128, 1),      # a decode projection (stream GEMV: no scratch needed)
    (1024, 32768, 4, 128, 8),     # x too large to stay resident: every row block split over many CTAs
    (1024, 11008, 4, 128, 1),     # few rows: the stream GEMV, one CTA per slab
    (1000, 1016, 8, 0, 3),        # ragged N and K, INT8 per channel, several tokens
    (8192, 32768, 4, 128, 1),     # long K
    (256, 512, 4, 128, 8),
])
def test_noalloc_matches_gemv_twice(N, K, bits, group, M):
    import torch
    qw, W = layer(N, K, bits, group, 41)
    xb = synth.make_activations(M, K, 41)
    x = to_dev_bf16(xb)
    ref = to_host_bits(tf.gemv(W, x))
    ref64 = tf_oracle.bf16_bits_to_f64(ref)
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        got = to_host_bits(_noalloc(W, x, y))
        check_close(got, ref64, f"noalloc {N}x{K} w{bits} g{group} M={M}")
    # and against the oracle, as every other GEMV test does
    check_close(got, tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb), "noalloc vs oracle")


@pytest.mark.parametrize("N,K,bits,group,M", [(1024, 768, 4, 32, 1), (4096, 4096, 4, 128, 1), (300, 256, 4, 32, 5)])
def test_noalloc_allocates_nothing(N, K, bits, group, M):
    """After a first call (which may load the kernel and look up the scratch
    array's address), further calls leave the device's free memory and the
    caching allocator's reservation exactly as they were."""
    import torch
    _, W = layer(N, K, bits, group, 43)
    x = to_dev_bf16(synth.make_activations(M, K, 43))
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    _noalloc(W, x, y)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    for _ in range(20):
        _noalloc(W, x, y)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_reserved() == reserved0
    assert free1 == free0, f"device free memory changed by {free0 - free1} bytes"
