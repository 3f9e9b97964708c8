"""Failure detection on the GPU without a fault: every wait in the kernels is
bounded, and a kernel whose wait runs out records a code in the device error
word, writes nothing and exits with no copy in flight.

The test hook tf_test_stall_copies makes the producers issue no copies, so
that the first wait of each kernel family runs out after 1 ms: the stream
GEMV (0x700), the tile and slab GEMVs (0x600, also behind tf_gemm at
M <= 8) and the GEMM (one of its role codes 0x100..0x500).  The next call,
with the hook off, must be correct and report no error: the context is
intact and no workspace was left dirty.
"""

import time

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
    tf.test_stall_copies(False)
    assert tf.device_error() == 0


CASES = [
    # (call, N, K, bits, group, M, expected codes)
    ("gemv", 4096, 4096, 4, 128, 1, {0x700}),           # stream GEMV
    ("gemv", 3000, 2048, 8, 0, 3, {0x700}),
    ("gemv", 1024, 2048, 4, 128, 1, {0x700}),           # stream GEMV, one CTA per slab
    ("gemv", 1024, 768, 4, 32, 1, {0x600}),             # tile GEMV (K < 1024)
    ("gemv", 4096, 2048, 4, 32, 1, {0x600}),            # slab GEMV (groups of 32)
    ("gemv_noalloc", 1024, 768, 4, 32, 1, {0x600}),     # tile GEMV on the fixed scratch array
    ("gemm", 4096, 4096, 4, 128, 256, {0x100, 0x200, 0x300, 0x400, 0x500}),
    ("gemm", 2048, 1024, 8, 0, 64, {0x100, 0x200, 0x300, 0x400, 0x500}),
    ("gemm", 2048, 1024, 8, 0, 4, {0x600}),             # M <= 8: tf_gemm on the slab GEMV
    ("gemm", 2048, 768, 8, 0, 4, {0x600}),              # and on the tile GEMV (K < 1024)
]


@pytest.mark.parametrize("call,N,K,bits,group,M,codes", CASES,
                         ids=[f"{c[0]}-{c[1]}x{c[2]}-w{c[3]}g{c[4]}-M{c[5]}" for c in CASES])
def test_wait_runs_out_and_context_survives(call, N, K, bits, group, M, codes):
    import torch
    qw, W = layer(N, K, bits, group, 61)
    xb = synth.make_activations(M, K, 61)
    x = to_dev_bf16(xb)
    fn = {"gemv": tf.gemv, "gemm": tf.gemm, "gemv_noalloc": tf.gemv_noalloc}[call]
    fn(W, x)  # the lazy set-up (attributes, workspace) outside the stalled call
    torch.cuda.synchronize()
    assert tf.device_error() == 0
    tf.test_stall_copies(True, 1000)
    try:
        y = torch.full((M, N), 5.0, dtype=torch.bfloat16, device="cuda")
        t = time.perf_counter()
        fn(W, x, y)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t
    finally:
        tf.test_stall_copies(False)
    code = tf.device_error()
    assert code in codes, hex(code)
    assert elapsed < 1.0, f"the bounded waits took {elapsed:.3f} s"
    assert bool((y == 5.0).all()), "a call whose waits ran out must not write its output"
    # the next call is correct and clean
    got = to_host_bits(fn(W, x))
    torch.cuda.synchronize()
    assert tf.device_error() == 0
    check_close(got, tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb),
                f"{call} after a stalled call")
