"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

import block_sparse_attention_08_gb300 as msa
from block_sparse_attention_08_gb300.binding import msa_config

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
OK, NULL, SHAPE, DTYPE, WORKSPACE, ALIGN = 0, 1, 2, 3, 4, 5


def _header_functions():
    names = set()
    for h in os.listdir(INCLUDE):
        if h.endswith(".h"):
            src = re.sub(r"/\*.*?\*/", "", open(os.path.join(INCLUDE, h)).read(), flags=re.S)
            names |= set(re.findall(r"\b(msa_[a-z0-9_]+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    return msa.load()


def test_every_declared_symbol_is_exported(lib):
    names = _header_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n


def _cfg(**kw):
    c = msa_config()
    assert msa.load().msa_config_default(ctypes.byref(c)) == OK
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_default_config_is_the_m3_topology(lib):
    c = _cfg()
    assert (c.num_q_heads, c.num_kv_heads, c.head_dim, c.num_index_heads, c.index_dim, c.block_size) == \
        (64, 4, 128, 4, 128, 128)
    assert (c.topk, c.init_blocks, c.local_blocks, c.index_dtype) == (16, 0, 1, 0)
    assert lib.msa_config_check(ctypes.byref(c)) == OK


@pytest.mark.parametrize("kw,code", [
    (dict(num_q_heads=32), SHAPE), (dict(num_kv_heads=8), SHAPE), (dict(head_dim=64), SHAPE),
    (dict(block_size=64), SHAPE), (dict(index_dim=64), SHAPE), (dict(topk=0), SHAPE), (dict(topk=17), SHAPE),
    (dict(init_blocks=-1), SHAPE), (dict(init_blocks=10, local_blocks=7), SHAPE), (dict(index_dtype=2), DTYPE),
])
def test_config_rejections(lib, kw, code):
    assert lib.msa_config_check(ctypes.byref(_cfg(**kw))) == code


def test_workspace_sizes(lib):
    c = _cfg()
    out = ctypes.c_size_t()
    assert lib.msa_workspace_size(ctypes.byref(c), 0, 64, 512, ctypes.byref(out)) == OK
    assert out.value >= 64 * 4 * 512 * 4 + 256
    small = out.value
    assert lib.msa_workspace_size(ctypes.byref(c), 0, 128, 512, ctypes.byref(out)) == OK
    assert out.value > small
    assert lib.msa_workspace_size(ctypes.byref(c), 1, 16384, 128, ctypes.byref(out)) == OK
    assert lib.msa_workspace_size(ctypes.byref(c), 2, 2 * 32768, 2, ctypes.byref(out)) == OK
    assert lib.msa_workspace_size(ctypes.byref(c), 7, 16, 1, ctypes.byref(out)) == SHAPE
    assert lib.msa_workspace_size(ctypes.byref(c), 0, 0, 1, ctypes.byref(out)) == SHAPE
    assert lib.msa_workspace_size(None, 0, 1, 1, ctypes.byref(out)) == NULL


FAKE = 0x10000  # 256-byte aligned address never dereferenced: every call below fails validation first


def test_select_decode_validation(lib):
    c = _cfg()
    f = lib.msa_select_blocks_decode
    ws_need = ctypes.c_size_t()
    lib.msa_workspace_size(ctypes.byref(c), 0, 4, 64, ctypes.byref(ws_need))
    args = [FAKE, FAKE, FAKE, FAKE, None, 4, 64, 4 * 8192, FAKE, FAKE, ws_need.value, None]
    assert f(ctypes.byref(_cfg(topk=17)), *args) == SHAPE
    assert f(ctypes.byref(c), None, *args[1:]) == NULL
    a = list(args); a[2] = None
    assert f(ctypes.byref(c), *a) == NULL
    a = list(args); a[3] = None; a[4] = None
    assert f(ctypes.byref(c), *a) == NULL           # neither page table nor cu_seqlens_k
    a = list(args); a[5] = 0
    assert f(ctypes.byref(c), *a) == SHAPE          # batch 0
    a = list(args); a[3] = FAKE; a[7] = 1000
    assert f(ctypes.byref(c), *a) == SHAPE          # paged pool not a whole number of pages
    a = list(args); a[0] = FAKE + 8
    assert f(ctypes.byref(c), *a) == ALIGN
    a = list(args); a[10] = ws_need.value - 1
    assert f(ctypes.byref(c), *a) == WORKSPACE
    a = list(args); a[9] = FAKE + 16
    assert f(ctypes.byref(c), *a) == WORKSPACE      # workspace not 256-byte aligned
    a = list(args); a[9] = None
    assert f(ctypes.byref(c), *a) == WORKSPACE


def test_attend_and_prefill_validation(lib):
    c = _cfg()
    assert lib.msa_sparse_attend_decode(ctypes.byref(c), FAKE, FAKE, FAKE, None, FAKE, None, FAKE, 4, 64,
                                        32768, ctypes.c_float(0.1), FAKE, FAKE, 1 << 30, None) == NULL
    assert lib.msa_sparse_attend_decode(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 4, 64,
                                        32768, ctypes.c_float(0.1), FAKE + 4, FAKE, 1 << 30, None) == ALIGN
    bad = _cfg(index_dtype=5)  # neither bf16 nor E4M3
    assert lib.msa_select_blocks_prefill(ctypes.byref(bad), FAKE, FAKE, FAKE, 1, 128, 128, FAKE, FAKE, 1 << 30,
                                         None) == DTYPE
    assert lib.msa_select_blocks_prefill(ctypes.byref(c), FAKE, FAKE, FAKE, 0, 128, 128, FAKE, FAKE, 1 << 30,
                                         None) == SHAPE
    assert lib.msa_select_blocks_prefill(ctypes.byref(c), FAKE, FAKE, FAKE, 1, 128, 300, FAKE, FAKE, 1 << 30,
                                         None) == SHAPE   # max_seqlen > tokens
    assert lib.msa_sparse_attend_prefill(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, None, 1, 128, 128,
                                         ctypes.c_float(0.1), FAKE, FAKE, 1 << 30, None) == NULL
    assert lib.msa_sparse_attend_prefill(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 128,
                                         ctypes.c_float(0.1), FAKE, FAKE, 16, None) == WORKSPACE


def test_backward_and_lse_validation(lib):
    c = _cfg()
    f = ctypes.c_float(0.1)
    # lse variant: a null lse
    assert lib.msa_sparse_attend_prefill_lse(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 128, f, FAKE,
                                             None, FAKE, 1 << 30, None) == NULL
    # backward: a null gradient, a misaligned output, a workspace too small
    args = [FAKE, FAKE, FAKE, FAKE, FAKE, 1, 128, 128, f, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE]
    bad = list(args)
    bad[11] = None  # grad_out
    assert lib.msa_sparse_attend_prefill_backward(ctypes.byref(c), *bad, FAKE, 1 << 30, None) == NULL
    bad = list(args)
    bad[12] = FAKE + 8  # dq
    assert lib.msa_sparse_attend_prefill_backward(ctypes.byref(c), *bad, FAKE, 1 << 30, None) == ALIGN
    assert lib.msa_sparse_attend_prefill_backward(ctypes.byref(c), *args, FAKE, 16, None) == WORKSPACE
    # its workspace: a mode of its own, smaller than the forward's
    fwd, bwd = ctypes.c_size_t(), ctypes.c_size_t()
    assert lib.msa_workspace_size(ctypes.byref(c), 1, 16384, 128, ctypes.byref(fwd)) == OK
    assert lib.msa_workspace_size(ctypes.byref(c), 3, 16384, 128, ctypes.byref(bwd)) == OK
    assert 0 < bwd.value < fwd.value


def test_pack_validation(lib):
    n, t, m, bad = ctypes.c_int(), ctypes.c_int64(), ctypes.c_int(), ctypes.c_int64()
    r = lib.msa_pack_metadata(FAKE, 0, 5, FAKE, FAKE, ctypes.byref(n), ctypes.byref(t), ctypes.byref(m),
                              ctypes.byref(bad), FAKE, 1 << 20, None)
    assert r == 7 and bad.value == -1                     # empty map
    r = lib.msa_pack_metadata(FAKE, 65536, 65536, FAKE, FAKE, ctypes.byref(n), ctypes.byref(t), ctypes.byref(m),
                              ctypes.byref(bad), FAKE, 1 << 20, None)
    assert r == 7                                        # past int32
    assert lib.msa_pack(FAKE, FAKE, 10, 24, FAKE, None) == SHAPE
    assert lib.msa_pack(None, FAKE, 10, 32, FAKE, None) == NULL
    assert lib.msa_unpack(FAKE, FAKE, 10, 5, 32, FAKE, None) == SHAPE


def test_bounded_wait_check_validation(lib):
    waits = (ctypes.c_int64 * 2)()
    assert lib.msa_check_bounded_wait(None, None, waits) == NULL
    assert lib.msa_check_bounded_wait(FAKE, None, None) == NULL
    assert lib.msa_check_bounded_wait(FAKE + 16, None, waits) == WORKSPACE


def test_index_produce_validation(lib):
    c = _cfg()
    # prefill: neither a packed key output nor a cache; a cache without a page table
    assert lib.msa_index_produce_prefill(ctypes.byref(c), FAKE, FAKE, FAKE, 1, 128, FAKE, None, None, None, 0, 0,
                                         FAKE, 256, None) == NULL
    assert lib.msa_index_produce_prefill(ctypes.byref(c), FAKE, FAKE, FAKE, 1, 128, FAKE, None, FAKE, None, 1,
                                         128, FAKE, 256, None) == NULL
    # a cache whose slot count is not a whole number of pages; a misaligned output; a small workspace
    assert lib.msa_index_produce_prefill(ctypes.byref(c), FAKE, FAKE, FAKE, 1, 128, FAKE, None, FAKE, FAKE, 1,
                                         100, FAKE, 256, None) == SHAPE
    assert lib.msa_index_produce_prefill(ctypes.byref(c), FAKE, FAKE, FAKE, 1, 128, FAKE + 8, FAKE, None, None,
                                         0, 0, FAKE, 256, None) == ALIGN
    assert lib.msa_index_produce_prefill(ctypes.byref(c), FAKE, FAKE, FAKE, 1, 128, FAKE, FAKE, None, None, 0, 0,
                                         FAKE, 128, None) == WORKSPACE
    bad = _cfg(index_dtype=7)
    assert lib.msa_index_produce_prefill(ctypes.byref(bad), FAKE, FAKE, FAKE, 1, 128, FAKE, FAKE, None, None, 0,
                                         0, FAKE, 256, None) == DTYPE
    # decode: no cache; no geometry; a bad batch
    assert lib.msa_index_produce_decode(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, None, 4, 8, 1024, FAKE, None,
                                        FAKE, 256, None) == NULL
    assert lib.msa_index_produce_decode(ctypes.byref(c), FAKE, FAKE, FAKE, None, None, 4, 8, 1024, FAKE, FAKE,
                                        FAKE, 256, None) == NULL
    assert lib.msa_index_produce_decode(ctypes.byref(c), FAKE, FAKE, FAKE, FAKE, None, 0, 8, 1024, FAKE, FAKE,
                                        FAKE, 256, None) == SHAPE


def test_status_strings(lib):
    for s in range(8):
        assert lib.msa_status_string(s)
    assert lib.msa_status_string(99) == b"unknown status"


def test_cuda_error_reporting(lib):
    # no call of this thread has failed in CUDA; the text is the runtime's
    # own for a code (a table lookup: no device is touched)
    assert lib.msa_last_cuda_error() == 0
    assert lib.msa_cuda_error_string(0) == b"no error"
    assert lib.msa_cuda_error_string(1) == b"invalid argument"
    # argument errors are caught before any CUDA call and leave it unchanged
    assert lib.msa_check_bounded_wait(None, None, None) == NULL
    assert lib.msa_last_cuda_error() == 0


def test_cuda_error_text_in_binding_errors():
    # the binding appends the CUDA error text to MSA_ERR_CUDA failures
    from block_sparse_attention_08_gb300 import binding
    assert binding.MSA_ERR_CUDA == 6
    e = binding.MsaError("msa_x", 6, "CUDA error: invalid argument (cudaError 1)")
    assert "invalid argument" in str(e) and e.status == 6
