"""C ABI checks that need no GPU: the library loads, exports every symbol include/tq.h
declares, its host-side constants agree with the oracle's independent computation, and
invalid arguments are rejected with error codes before anything is launched."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle.turboquant as o
from kv_cache_quantization_gb300 import _binding as B
from kv_cache_quantization_gb300.synth import gaussian_matrix

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tq.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        from kv_cache_quantization_gb300 import build
        build.build()
    return B.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_header_symbols_exported(lib):
    names = declared_functions()
    assert len(names) >= 14
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\S+)$", out, flags=re.M))
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    not_bound = [n for n in names if n not in B.SIGNATURES]
    assert not not_bound, f"declared but not bound in Python: {not_bound}"
    for n in names:
        assert hasattr(lib, n)


def test_status_strings(lib):
    for s in range(7):
        assert B.tq_status_string(s).startswith("TQ_")
    assert "sm_103a" in B.tq_version()


@pytest.mark.parametrize("bits", [1, 2, 3, 4])
def test_codebook_matches_oracle(lib, bits):
    c = np.zeros(1 << bits)
    assert B.tq_lloyd_max_codebook(128, bits, c.ctypes.data) == B.TQ_OK
    ref, _ = o.lloyd_max_codebook(128, bits)
    np.testing.assert_allclose(c, ref, rtol=0, atol=1e-12)
    assert np.all(c[:len(c) // 2] == -c[::-1][:len(c) // 2])


def test_rotation_matches_oracle(lib):
    g = gaussian_matrix(42)
    pi = np.zeros((128, 128))
    assert B.tq_rotation_from_gaussian(128, g.ctypes.data, pi.ctypes.data) == B.TQ_OK
    np.testing.assert_allclose(pi, o.rotation_from_gaussian(g), rtol=0, atol=1e-12)


def test_code_bytes(lib):
    assert B.tq_code_bytes(B.TQ_PROD, 3) == 56 and B.tq_code_bytes(B.TQ_PROD, 4) == 72
    assert B.tq_code_bytes(B.TQ_MSE, 4) == 68 and B.tq_code_bytes(B.TQ_MSE, 2) == 36
    assert B.tq_code_bytes(B.TQ_PROD, 1) == 0 and B.tq_code_bytes(B.TQ_MSE, 5) == 0


def test_bounded_wait_check_rejects_limits_out_of_range(lib):
    assert B.tq_check_bounded_wait(0, None) == B.TQ_ERR_INVALID_ARG
    assert B.tq_check_bounded_wait(1000001, None) == B.TQ_ERR_INVALID_ARG


def test_invalid_arguments_rejected(lib):
    pi = np.eye(128)
    c = np.array([-0.1, 0.1])
    h = ctypes.c_void_p()
    # unsupported head dim / bit width, missing pointers, unsorted levels
    assert B.tq_codec_create(64, B.TQ_MSE, 1, pi, None, c, h) == B.TQ_ERR_UNSUPPORTED
    assert B.tq_codec_create(128, B.TQ_MSE, 7, pi, None, c, h) == B.TQ_ERR_UNSUPPORTED
    assert B.tq_codec_create(128, B.TQ_PROD, 2, pi, None, c, h) == B.TQ_ERR_INVALID_ARG
    assert B.tq_codec_create(128, B.TQ_MSE, 1, None, None, c, h) == B.TQ_ERR_INVALID_ARG
    assert B.tq_codec_create(128, B.TQ_MSE, 1, pi, None, c[::-1].copy(), h) == B.TQ_ERR_INVALID_ARG
    assert B.tq_lloyd_max_codebook(128, 5, c.ctypes.data) == B.TQ_ERR_INVALID_ARG
    assert B.tq_rotation_from_gaussian(128, None, None) == B.TQ_ERR_INVALID_ARG
    # calls with a null codec
    empty = B.tq_prod_cache(0, 0, 0, 0)
    assert B.tq_quantize_prod(None, 16, B.TQ_BF16, 1, 1, 1, 0, 0, 128, None, None, empty, 64,
                              None) == B.TQ_ERR_INVALID_ARG
    assert B.tq_quantize_mse(None, 16, B.TQ_BF16, 1, 1, 1, 0, 0, 128, None, None,
                             B.tq_mse_cache(0, 0), 64, None) == B.TQ_ERR_INVALID_ARG
    assert B.tq_prod_scores(None, 16, 1, 128, empty, 64, 1, 16, 1, None) == B.TQ_ERR_INVALID_ARG
    # descriptors
    d = B.tq_attn_desc(1, 28, 4, 128, 32768, 32768, 0, 0.0, B.TQ_BF16, B.TQ_F32)
    bad = [B.tq_attn_desc(1, 28, 4, 64, 32768, 32768, 0, 0.0, B.TQ_BF16, B.TQ_F32),   # d
           B.tq_attn_desc(1, 28, 5, 128, 32768, 32768, 0, 0.0, B.TQ_BF16, B.TQ_F32),  # Hq % Hkv
           B.tq_attn_desc(1, 36, 4, 128, 32768, 32768, 0, 0.0, B.TQ_BF16, B.TQ_F32),  # G = 9
           B.tq_attn_desc(1, 28, 4, 128, 1000, 1000, 0, 0.0, B.TQ_BF16, B.TQ_F32),    # capacity
           B.tq_attn_desc(1, 28, 4, 128, 1024, 2048, 0, 0.0, B.TQ_BF16, B.TQ_F32),    # max len
           B.tq_attn_desc(1, 28, 4, 128, 1024, 1024, 0, 0.0, 7, B.TQ_F32)]            # dtype
    for bd in bad:
        assert B.tq_decode_workspace_bytes(bd) == 0
    assert B.tq_decode_attention(bad[0], None, None, 16, empty, B.tq_mse_cache(0, 0), 16, 16, 256,
                                 1 << 20, None) == B.TQ_ERR_UNSUPPORTED
    assert B.tq_decode_attention(d, None, None, 16, empty, B.tq_mse_cache(0, 0), 16, 16, 256,
                                 1 << 20, None) == B.TQ_ERR_INVALID_ARG
    assert B.tq_decode_attention_asym(d, None, 16, 16, B.tq_mse_cache(0, 0), 16, 16, 16, 16, 16,
                                      256, 1 << 20, None) == B.TQ_ERR_INVALID_ARG


def test_struct_layouts_match_header(tmp_path):
    """The binding's ctypes structs have the sizes and field offsets that the C header gives
    (compiled here with the host C compiler)."""
    src = tmp_path / "layout.c"
    src.write_text(
        "#include <stddef.h>\n#include <stdio.h>\n#include \"tq.h\"\n"
        "int main(void) {\n"
        "  printf(\"%zu %zu %zu %zu %zu %zu %zu %zu\\n\", sizeof(tq_pages),\n"
        "         offsetof(tq_pages, num_pages), sizeof(tq_prod_cache),\n"
        "         offsetof(tq_prod_cache, pages), sizeof(tq_mse_cache),\n"
        "         offsetof(tq_mse_cache, pages), sizeof(tq_attn_desc),\n"
        "         offsetof(tq_attn_desc, out_dtype));\n"
        "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True,
                                          check=True).stdout.split()]
    want = [ctypes.sizeof(B.tq_pages), B.tq_pages.num_pages.offset,
            ctypes.sizeof(B.tq_prod_cache), B.tq_prod_cache.pages.offset,
            ctypes.sizeof(B.tq_mse_cache), B.tq_mse_cache.pages.offset,
            ctypes.sizeof(B.tq_attn_desc), B.tq_attn_desc.out_dtype.offset]
    assert got == want


def test_pages_host_object():
    """api.Pages: the table's shape gives the pages per sequence and the capacity, the C struct
    points at the table, and tables that are not int32 [batch, max_pages] are refused."""
    import torch

    from kv_cache_quantization_gb300 import api
    t = torch.tensor([[3, 1, -1], [0, 2, -1]], dtype=torch.int32)
    p = api.Pages(t, 64, 4)
    assert p.max_pages == 3 and p.capacity == 192
    c = p.c().contents
    assert (c.block_table, c.max_pages, c.page_tokens, c.num_pages) == (t.data_ptr(), 3, 64, 4)
    with pytest.raises(ValueError):
        api.Pages(t.long(), 64, 4)
    with pytest.raises(ValueError):
        api.Pages(t[0], 64, 4)
