"""The C ABI: libmla.so builds, loads and exports every call include/mla.h declares;
host-side validation rejects bad arguments before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mla.h")


@pytest.fixture(scope="module")
def L():
    from mla_attention_gb300 import build as b
    b.build()
    from mla_attention_gb300 import _lib
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mla_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for need in ["mla_prefill", "mla_prefill_split", "mla_decode", "mla_sparse", "mla_merge_lse",
                 "mla_prefill_workspace_size", "mla_decode_workspace_size", "mla_sparse_workspace_size",
                 "mla_prefill_split_workspace_size", "mla_last_error_string", "mla_check_device_status"]:
        assert need in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"libmla.so does not export {name}"


def test_binding_covers_every_declared_symbol():
    from mla_attention_gb300 import _lib
    assert set(declared_functions()) <= set(_lib.exported_symbols())


def test_status_strings_and_version(L):
    assert L.mla_version() >= 100
    assert L.mla_status_string(0) == b"MLA_OK"
    assert L.mla_status_string(4) == b"MLA_ERR_TIMEOUT"


def _prefill(L, **kw):
    a = dict(q=None, sT=128 * 576, sH=576, kv=None, skv=576, T=4, H=128, Tkv=4, dk=576, dv=512, scale=0.07,
             causal=1, qp=0, kp=0, kvv=-1, po=None, pl=None, out=None, lse=None, ws=None, wsb=0, st=None)
    a.update(kw)
    return L.mla_prefill(a["q"], a["sT"], a["sH"], a["kv"], a["skv"], a["T"], a["H"], a["Tkv"], a["dk"], a["dv"],
                         a["scale"], a["causal"], a["qp"], a["kp"], a["kvv"], a["po"], a["pl"], a["out"], a["lse"],
                         a["ws"], a["wsb"], a["st"])


def test_prefill_validation(L):
    fake = ctypes.c_void_p(1 << 20)
    # only the DeepSeek geometry is built
    assert _prefill(L, dk=192, dv=128, ws=fake, wsb=256) == 2
    # V must be narrower than K
    assert _prefill(L, dk=512, dv=576, ws=fake, wsb=256) == 1
    # prev pair is both-or-neither
    assert _prefill(L, po=fake, ws=fake, wsb=256) == 1
    # workspace required
    assert _prefill(L) == 6
    # kv_valid beyond Tkv
    assert _prefill(L, kvv=9, ws=fake, wsb=256) == 1
    # T * H of 2^31 or more: output rows are signed 32-bit tensor-map coordinates
    assert _prefill(L, T=1 << 24, Tkv=0, kvv=0, q=fake, out=fake, lse=fake, ws=fake, wsb=1 << 40) == 1
    assert b"T * H" in L.mla_last_error_string()
    # T = 0 is a no-op (no launch, no CUDA call)
    assert _prefill(L, T=0, ws=fake, wsb=256) == 0
    assert L.mla_last_error_string() == b""  # a successful call leaves no error text


def test_sparse_and_split_validation(L):
    fake = ctypes.c_void_p(1 << 20)
    # B must be 1; softmax_scale must be positive; H <= 128
    assert L.mla_sparse(fake, fake, fake, fake, fake, 2, 4, 8, 16, 128, 0.1, fake, None, fake, 256, None) == 1
    assert L.mla_sparse(fake, fake, fake, fake, fake, 1, 4, 8, 16, 128, -0.1, fake, None, fake, 256, None) == 1
    assert L.mla_sparse(fake, fake, fake, fake, fake, 1, 4, 8, 256, 128, 0.1, fake, None, fake, 256, None) == 2
    seq = (ctypes.c_int32 * 2)(4, 4)
    # head_num % kv_head_num
    assert L.mla_prefill_split(fake, fake, fake, fake, fake, seq, 1, 2, 6, 4, 0.1, 1, None, None, fake, fake,
                               fake, 256, None) == 1
    # mask type
    assert L.mla_prefill_split(fake, fake, fake, fake, fake, seq, 1, 2, 4, 4, 0.1, 3, None, None, fake, fake,
                               fake, 256, None) == 1


def test_decode_and_merge_validation(L):
    fake = ctypes.c_void_p(1 << 20)
    assert L.mla_decode(fake, fake, 8, 48, fake, 4, fake, 2, 128, 0.1, 0, fake, None, fake, 1 << 30, None) == 1
    assert L.mla_decode(fake, fake, 8, 64, fake, 4, fake, 2, 256, 0.1, 0, fake, None, fake, 1 << 30, None) == 2
    assert L.mla_decode(fake, fake, 8, 64, fake, 4, fake, 2, 128, 0.1, 0, fake, None, fake, 16, None) == 6
    # num_pages * page_size of 2^31 or more: cache rows are signed 32-bit tensor-map coordinates
    assert L.mla_decode(fake, fake, 1 << 25, 64, fake, 4, fake, 2, 128, 0.1, 0, fake, None, fake, 1 << 30, None) == 1
    assert b"num_pages * page_size" in L.mla_last_error_string()
    assert L.mla_merge_lse(fake, fake, fake, fake, fake, fake, 4, 2, 12, None) == 1
    assert L.mla_merge_lse(None, None, None, None, None, None, 0, 2, 16, None) == 0


def test_workspace_sizes(L):
    assert L.mla_prefill_workspace_size(8192, 128) >= 256
    # decode partials: (B + pairs) slots x H x (512 + 1) fp32
    assert L.mla_decode_workspace_size(64, 128, 76) >= (64 + 76) * 128 * 513 * 4


def test_bench_flop_accounting():
    """The bench counts unmasked (token, key) pairs per KV chunk; the four chunks of the
    8192-token causal prefill must add up to T (T + 1) / 2, and chunk j (keys 2048 j ..
    2048 j + 2047) is a causal triangle plus full rows for the later tokens."""
    import bench
    T, C = bench.T_TOTAL, bench.CHUNK
    pairs = bench.chunk_pairs()
    assert sum(pairs) == T * (T + 1) // 2
    for j, n in enumerate(pairs):
        assert n == C * (C + 1) // 2 + (T - C * (j + 1)) * C
    assert bench.FLOP_PER_PAIR == 2 * 128 * (576 + 512)
