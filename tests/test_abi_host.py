"""Host-side tests of libtf through its C ABI (no GPU needed).

The library must load and export every function include/tf.h declares; the
C++ pre-tiling must produce exactly the blob the reference layout defines;
its inverse must be exact; invalid arguments must come back as status codes.
"""

import ctypes
import subprocess

import numpy as np
import pytest

import gemv_tf_prepack_gb300 as tf
from gemv_tf_prepack_gb300 import synth
from oracle import layout as L


@pytest.fixture(scope="session", autouse=True)
def built_library():
    from gemv_tf_prepack_gb300 import build as b
    b.build()
    return tf.lib()


def test_exports_every_declared_symbol():
    decl = tf.header_declarations()
    assert len(decl) >= 11
    out = subprocess.run(["nm", "-D", "--defined-only", tf.lib_path], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [d for d in decl if d not in exported]
    assert not missing, missing
    lib = tf.lib()
    for d in decl:
        getattr(lib, d)
    assert tf.version() == 6


@pytest.mark.parametrize("N,K,bits,group", [
    (256, 512, 4, 128), (200, 192, 4, 64), (136, 200, 8, 0), (64, 96, 4, 32),
    (130, 256, 8, 128), (8, 8, 4, 0), (128, 1024, 4, 256), (300, 384, 8, 64), (72, 96, 8, 32),
    (200, 1003, 4, 0), (130, 77, 8, 0), (17, 5, 4, 0), (33, 3, 8, 0),  # K % 8 != 0, per channel
])
def test_prepack_matches_reference_layout(N, K, bits, group):
    qw = synth.make_weights(N, K, bits, group, 5)
    ref = L.prepack(qw.qweight, qw.scales, qw.zeros, N, K, bits, group)
    got = tf.prepack(qw.qweight, qw.scales, qw.zeros, N, K, bits, group)
    assert got.size == ref.size == tf.prepack_size(N, K, bits, group)
    np.testing.assert_array_equal(got, ref)
    qw2, s2, z2, n2, k2, b2, g2 = tf.unprepack(got)
    assert (n2, k2, b2, g2) == (N, K, bits, group)
    np.testing.assert_array_equal(qw2, qw.qweight)
    np.testing.assert_array_equal(s2, qw.scales)
    np.testing.assert_array_equal(z2, qw.zeros)


def test_prepack_decode_shape_round_trip():
    N, K = 4096, 4096
    qw = synth.make_weights(N, K, 4, 128, 2)
    blob = tf.prepack(qw.qweight, qw.scales, qw.zeros, N, K, 4, 128)
    r = tf.unprepack(blob)
    np.testing.assert_array_equal(r[0], qw.qweight)
    np.testing.assert_array_equal(r[1], qw.scales)
    np.testing.assert_array_equal(r[2], qw.zeros)


def test_prepack_sizes():
    assert tf.prepack_size(32768, 32768, 4, 128) == 64 + 2048 * 256 * 1072
    assert tf.prepack_size(8192, 8192, 8, 0) == 64 + 512 * 64 * 2112
    assert tf.prepack_size(4096, 4096, 4, 64) == 64 + 32 * 32 * 8832


def _rc(fn, *args):
    return fn(*args)


def test_invalid_arguments_return_codes():
    lib = tf.lib()
    sz = ctypes.c_size_t()
    assert lib.tf_prepack_size(0, 128, 4, 128, ctypes.byref(sz)) == -1
    assert lib.tf_prepack_size(128, 100, 4, 0, ctypes.byref(sz)) == 0        # K % 8 != 0: per channel only
    assert sz.value == 64 + 8 * 1 * 1072
    assert lib.tf_prepack_size(128, 256, 4, 96, ctypes.byref(sz)) == -2      # group 96
    assert lib.tf_prepack_size(128, 192, 4, 128, ctypes.byref(sz)) == -1     # K % g
    assert lib.tf_prepack_size(32769, 128, 4, 128, ctypes.byref(sz)) == -2   # > 32K
    assert lib.tf_prepack_size(128, 128, 3, 128, ctypes.byref(sz)) == -2     # bits
    assert lib.tf_prepack_size(32768, 32768, 8, 0, ctypes.byref(sz)) == 0
    assert lib.tf_prepack_size(128, 128, 4, 128, None) == -1
    # zeros out of range for INT4
    qw = np.zeros((8, 16), np.uint32)
    s = np.zeros((8, 1), np.uint16)
    z = np.full((8, 1), 16, np.uint8)
    out = np.zeros(tf.prepack_size(8, 128, 4, 128), np.uint8)
    assert lib.tf_prepack(qw.ctypes.data, s.ctypes.data, z.ctypes.data, 8, 128, 4, 128,
                          out.ctypes.data, out.size) == -1
    assert lib.tf_prepack(qw.ctypes.data, s.ctypes.data, z.ctypes.data, 8, 128, 4, 128,
                          out.ctypes.data, out.size - 1) == -1
    # corrupted header
    z[:] = 3
    assert lib.tf_prepack(qw.ctypes.data, s.ctypes.data, z.ctypes.data, 8, 128, 4, 128,
                          out.ctypes.data, out.size) == 0
    bad = out.copy()
    bad[0] ^= 1
    with pytest.raises(tf.TFError) as e:
        tf.unprepack(bad)
    assert e.value.status == -5
    short = out[:-16]
    with pytest.raises(tf.TFError):
        tf.unprepack(short)
    for code in range(-8, 1):
        assert lib.tf_status_string(code)
    assert lib.tf_status_string(-8).decode().startswith("TF_ERR_SCRATCH_LIMIT")
    assert lib.tf_status_string(-5).decode().startswith("TF_ERR_BAD_BLOB")


def test_device_calls_validate_before_touching_the_gpu():
    """Argument errors are reported without any CUDA call."""
    lib = tf.lib()
    blob = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    size = tf.prepack_size(256, 512, 4, 128)
    x = ctypes.c_void_p(8192)
    y = ctypes.c_void_p(16384)
    # wrong blob size
    assert lib.tf_gemv(blob, size - 16, 256, 512, 4, 128, x, y, 1, None, 0, None) == -5
    # misaligned blob
    assert lib.tf_gemv(ctypes.c_void_p(4100), size, 256, 512, 4, 128, x, y, 1, None, 0, None) == -3
    # M out of range
    assert lib.tf_gemv(blob, size, 256, 512, 4, 128, x, y, 9, None, 0, None) == -2
    assert lib.tf_gemv(blob, size, 256, 512, 4, 128, x, y, 0, None, 0, None) == -1
    assert lib.tf_gemm(blob, size, 256, 512, 4, 128, x, y, 0, None, 0, None) == -1
    assert lib.tf_gemm(blob, size, 256, 512, 4, 128, ctypes.c_void_p(8194), y, 4, None, 0, None) == -3
    assert lib.tf_gemm(blob, size, 256, 512, 4, 128, x, y, 4, ctypes.c_void_p(8200), 64, None) == -3
    # the bias variants: an odd bias address, and the same checks as the plain calls
    odd = ctypes.c_void_p(20001)
    assert lib.tf_gemv_bias(blob, size, 256, 512, 4, 128, x, odd, y, 1, None, 0, None) == -3
    assert lib.tf_gemm_bias(blob, size, 256, 512, 4, 128, x, odd, y, 4, None, 0, None) == -3
    assert lib.tf_gemv_bias(blob, size, 256, 512, 4, 128, x, None, y, 9, None, 0, None) == -2
    assert lib.tf_gemv_bias(blob, size - 16, 256, 512, 4, 128, x, None, y, 1, None, 0, None) == -5
    assert lib.tf_gemm_bias(blob, size, 256, 512, 4, 128, x, None, None, 4, None, 0, None) == -1
    assert lib.tf_dequant(None, size, 256, 512, 4, 128, y, None) == -1
    assert lib.tf_dequant(blob, size, 256, 512, 4, 96, y, None) == -2
    # the fused epilogues: the layer's checks, then the epilogue's own
    for fn in (lib.tf_gemv_silu_gate, lib.tf_gemm_silu_gate):
        assert fn(blob, size - 16, 256, 512, 4, 128, x, None, y, 1, None, 0, None) == -5
        assert fn(blob, size, 256, 512, 4, 128, x, None, None, 1, None, 0, None) == -1
        assert fn(blob, size, 256, 512, 4, 128, x, odd, y, 1, None, 0, None) == -3
        assert fn(blob, size, 256, 512, 4, 128, x, None, ctypes.c_void_p(16385), 1, None, 0, None) == -3
    size_n = tf.prepack_size(264, 512, 4, 128)  # N = 264: not a multiple of 16
    assert lib.tf_gemv_silu_gate(blob, size_n, 264, 512, 4, 128, x, None, y, 1, None, 0, None) == -1
    assert lib.tf_gemm_silu_gate(blob, size_n, 264, 512, 4, 128, x, None, y, 1, None, 0, None) == -1
    assert lib.tf_gemv_silu_gate(blob, size, 256, 512, 4, 128, x, None, y, 9, None, 0, None) == -2
    q, k, v = ctypes.c_void_p(16384), ctypes.c_void_p(24576), ctypes.c_void_p(32768)
    for fn in (lib.tf_gemv_qkv, lib.tf_gemm_qkv):
        assert fn(blob, size, 256, 512, 4, 128, x, None, q, k, v, 0, 64, 1, None, 0, None) == -1
        assert fn(blob, size, 256, 512, 4, 128, x, None, q, k, v, 128, -1, 1, None, 0, None) == -1
        assert fn(blob, size, 256, 512, 4, 128, x, None, q, k, v, 200, 57, 1, None, 0, None) == -1
        assert fn(blob, size, 256, 512, 4, 128, x, None, q, None, v, 128, 64, 1, None, 0, None) == -1
        assert fn(blob, size, 256, 512, 4, 128, x, None, q, k, None, 128, 64, 1, None, 0, None) == -1
        assert fn(blob, size, 256, 512, 4, 128, x, None, q, k, ctypes.c_void_p(32769), 128, 64, 1, None, 0,
                  None) == -3
        assert fn(blob, size - 16, 256, 512, 4, 128, x, None, q, k, v, 128, 64, 1, None, 0, None) == -5
    assert lib.tf_gemv_qkv(blob, size, 256, 512, 4, 128, x, None, q, k, v, 128, 64, 9, None, 0, None) == -2


def test_header_serves_a_plain_c_client(tmp_path):
    """include/tf.h compiles as C11 and a C program links against libtf and calls it."""
    import os
    import shutil
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda_inc = next((d for d in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda")
                     if d and os.path.exists(os.path.join(d, "include", "cuda_runtime_api.h"))), None)
    if cuda_inc is None:
        pytest.skip("cuda_runtime_api.h not found")
    pkg = os.path.dirname(tf.lib_path)
    src = tmp_path / "client.c"
    src.write_text(
        '#include "tf.h"\n#include <stdio.h>\n'
        "int main(void) {\n"
        "  size_t bytes = 0;\n"
        "  int rc = tf_prepack_size(4096, 4096, 4, 128, &bytes);\n"
        "  size_t unused = 0;\n"
        "  int bad = tf_prepack_size(4096, 4096, 3, 128, &unused);  /* 3-bit codes: unsupported */\n"
        '  printf("%d %d %zu %d %s\\n", tf_version(), rc, bytes, bad, tf_status_string(bad));\n'
        "  return rc;\n}\n")
    exe = tmp_path / "client"
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.dirname(tf.HEADER), "-I",
                    os.path.join(cuda_inc, "include"), str(src), "-o", str(exe), "-L", pkg, "-ltf",
                    "-Wl,-rpath," + pkg], check=True, capture_output=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    assert out[:4] == [str(tf.version()), "0", str(tf.prepack_size(4096, 4096, 4, 128)), "-2"]
    assert out[4] == "TF_ERR_UNSUPPORTED:"


def test_plain_c_client_packs_a_gate_up_layer(tmp_path):
    """A C11 program builds a gate/up blob with tf_prepack_gate_up and reads it
    back with tf_blob_info; the bytes equal the Python binding's."""
    import os
    import shutil
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda_inc = next((d for d in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda")
                     if d and os.path.exists(os.path.join(d, "include", "cuda_runtime_api.h"))), None)
    if cuda_inc is None:
        pytest.skip("cuda_runtime_api.h not found")
    F, K = 8, 24  # K % 8 == 0 here; per channel
    g = synth.make_weights(F, K, 4, 0, 11)
    u = synth.make_weights(F, K, 4, 0, 12)
    arrays = {"gq": g.qweight, "gs": g.scales, "gz": g.zeros, "uq": u.qweight, "us": u.scales, "uz": u.zeros}
    for name, a in arrays.items():
        np.ascontiguousarray(a).tofile(tmp_path / f"{name}.bin")
    size = tf.prepack_size(2 * F, K, 4, 0)
    src = tmp_path / "gate_up.c"
    src.write_text(
        '#include "tf.h"\n#include <stdio.h>\n#include <stdlib.h>\n'
        "static void* load(const char* path, size_t n) {\n"
        "  void* p = malloc(n); FILE* f = fopen(path, \"rb\");\n"
        "  if (!f || fread(p, 1, n, f) != n) exit(3);\n"
        "  fclose(f); return p;\n}\n"
        "int main(int argc, char** argv) {\n"
        "  (void)argc;\n"
        f"  const int F = {F}, K = {K};\n"
        "  char path[4096];\n"
        "#define LOAD(name, n) (snprintf(path, sizeof path, \"%s/%s.bin\", argv[1], name), load(path, n))\n"
        "  void* gq = LOAD(\"gq\", (size_t)F * (K / 8) * 4); void* uq = LOAD(\"uq\", (size_t)F * (K / 8) * 4);\n"
        "  uint16_t* gs = LOAD(\"gs\", (size_t)F * 2); uint16_t* us = LOAD(\"us\", (size_t)F * 2);\n"
        "  uint8_t* gz = LOAD(\"gz\", (size_t)F); uint8_t* uz = LOAD(\"uz\", (size_t)F);\n"
        f"  size_t bytes = {size};\n"
        "  unsigned char* blob = malloc(bytes);\n"
        "  int rc = tf_prepack_gate_up(gq, gs, gz, uq, us, uz, F, K, 4, 0, blob, bytes);\n"
        "  int n = 0, k = 0, bits = 0, group = -1;\n"
        "  int rc2 = tf_blob_info(blob, bytes, &n, &k, &bits, &group);\n"
        "  unsigned long sum = 0;\n"
        "  for (size_t i = 0; i < bytes; ++i) sum = sum * 31u + blob[i];\n"
        "  printf(\"%d %d %d %d %d %d %lu\\n\", rc, rc2, n, k, bits, group, sum);\n"
        "  return rc;\n}\n")
    exe = tmp_path / "gate_up"
    pkg = os.path.dirname(tf.lib_path)
    subprocess.run([cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.dirname(tf.HEADER), "-I",
                    os.path.join(cuda_inc, "include"), str(src), "-o", str(exe), "-L", pkg, "-ltf",
                    "-Wl,-rpath," + pkg], check=True, capture_output=True)
    out = subprocess.run([str(exe), str(tmp_path)], capture_output=True, text=True, check=True).stdout.split()
    want = tf.prepack_gate_up((g.qweight, g.scales, g.zeros), (u.qweight, u.scales, u.zeros), F, K, 4, 0)
    s = 0
    for b in want.tobytes():
        s = (s * 31 + b) % (1 << 64)
    assert out[:6] == ["0", "0", str(2 * F), str(K), "4", "0"]
    assert int(out[6]) == s
