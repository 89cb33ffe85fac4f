"""Small cases of every call of the library run through the guarded build (libmla_guard.so, path in
argv[1]), each compared with the oracle, with the status word read after each call: a guarded
check that fires (an access that would have left its buffer) fails the run.  Run as a child
process by tests/test_gpu_guarded.py, so that this process loads the guarded library and not the
default one.  Prints "guarded ok" and exits 0 when every case passes."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from mla_attention_gb300 import _lib  # noqa: E402

_lib.LIB_PATH = sys.argv[1]

import mla_attention_gb300 as lib  # noqa: E402
import oracle.mla_oracle as mo  # noqa: E402
from mla_attention_gb300 import inputs as gen  # noqa: E402
from tests.helpers import assert_lse_close, assert_out_close  # noqa: E402


def done():
    torch.cuda.synchronize()
    lib.check_device_status()   # raises MLAError on a guarded-check code (0x3000 | site)


def prefill_cases(d):
    for keys in (128, 64):
        lib.set_tile_keys(keys, keys)
        P = gen.prefill_inputs(T=300, H=16, Tkv=300, seed=5)   # several items per CTA pair, ragged tail
        po, pl = gen.prev_inputs(300, 16, 512, seed=6, lse_lo=1.0, lse_hi=6.0)
        out, lse = lib.mla_prefill(P.q.to(d), P.kv.to(d), P.scale, causal=True, q_pos0=100, kv_pos0=0,
                                   prev_out=po.to(d), prev_lse=pl.to(d))
        done()
        ro, rl = mo.mla_prefill(P.q, P.kv, P.scale, causal=True, q_pos0=100, kv_pos0=0, prev_out=po, prev_lse=pl)
        assert_out_close(out, ro)
        assert_lse_close(lse, rl)
    lib.set_tile_keys(0, 0)
    q_lens, kv_lens = [70, 0, 33], [70, 10, 150]
    g = torch.Generator().manual_seed(7)
    q = gen.randn_bf16((sum(q_lens), 8, 576), g)
    kv = gen.randn_bf16((sum(kv_lens), 576), g)
    cq = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(kv_lens)]).astype(np.int32)
    out, lse = lib.mla_prefill_varlen(q.to(d), kv.to(d), cq, ck, gen.SCALE_192, causal=True)
    done()
    for b in range(len(q_lens)):
        if q_lens[b]:
            qs, ks = slice(cq[b], cq[b + 1]), slice(ck[b], ck[b + 1])
            ro, rl = mo.mla_prefill(q[qs], kv[ks], gen.SCALE_192, causal=True, q_pos0=kv_lens[b] - q_lens[b])
            assert_out_close(out[qs], ro)
            assert_lse_close(lse[:, qs], rl)


def decode_cases(d):
    for keys in (128, 64):
        lib.set_tile_keys(keys, keys)
        D = gen.decode_inputs([300, 17, 0, 129], H=16, seed=8, page_size=16)
        out, lse = lib.mla_decode(D.q.to(d), D.cache.to(d), D.block_table.to(d), D.lens.to(d), D.scale,
                                  num_splits=5)
        done()
        ro, rl = mo.mla_decode(D.q, D.cache, D.block_table, D.lens, D.scale)
        assert_out_close(out, ro)
        assert_lse_close(lse, rl)
        g = torch.Generator().manual_seed(9)
        q2 = gen.randn_bf16((4, 2, 16, 576), g)
        sk = torch.randn((16,), generator=g).float()
        out, lse = lib.mla_decode_ex(q2.to(d), D.cache.to(d), D.block_table.to(d), D.lens.to(d), D.scale,
                                     sinks=sk.to(d), num_splits=3)
        done()
        ro, rl = mo.mla_decode_ex(q2, D.cache, D.block_table, D.lens, D.scale, sinks=sk)
        assert_out_close(out, ro)
        assert_lse_close(lse, rl)
    lib.set_tile_keys(0, 0)
    D = gen.decode_inputs([200, 70, 5], H=32, seed=10, page_size=64)
    c8 = (D.cache.float() / 0.37).to(torch.float8_e4m3fn)
    out, lse = lib.mla_decode_fp8(D.q.to(d), c8.to(d), 0.37, D.block_table.to(d), D.lens.to(d), D.scale)
    done()
    ro, rl = mo.mla_decode_fp8(D.q[:, None], c8, 0.37, D.block_table, D.lens, D.scale)
    assert_out_close(out, ro[:, 0])
    assert_lse_close(lse, rl[:, 0])
    out, lse = lib.mla_decode_noalloc(D.q.to(d), D.cache.to(d), D.block_table.to(d), D.lens.to(d), D.scale)
    torch.cuda.synchronize()
    ro, rl = mo.mla_decode(D.q, D.cache, D.block_table, D.lens, D.scale)
    assert_out_close(out, ro)


def sparse_cases(d):
    for keys, H in ((128, 128), (128, 16), (64, 16)):
        lib.set_tile_keys(keys, 0)
        SI = gen.sparse_inputs(90, 700, H, 256, 600, seed=11 + H)
        SI.topk[0, 0, 5] = -1
        SI.topk[0, 3, 128:256] = -1
        out, lse = lib.mla_sparse(SI.q_lift.to(d), SI.q_pe.to(d), SI.c_kv.to(d), SI.k_pe.to(d), SI.topk.to(d),
                                  SI.scale)
        done()
        ro, rl = mo.mla_sparse(SI.q_lift, SI.q_pe, SI.c_kv, SI.k_pe, SI.topk, SI.scale)
        assert_out_close(out, ro)
        assert_lse_close(lse, rl)
    lib.set_tile_keys(0, 0)


def split_merge_cases(d):
    si = gen.split_inputs([5, 130, 257], [5, 130, 257], 4, 2, seed=12, with_prev=True, prev_lse_range=(2.0, 5.0))
    out, lse = lib.mla_prefill_split(si.q_nope.to(d), si.q_pe.to(d), si.k_nope.to(d), si.k_pe.to(d), si.v.to(d),
                                     si.seq_len, si.head_num, si.kv_head_num, si.scale, 1,
                                     prev_out=si.prev_out.to(d), prev_lse=si.prev_lse.to(d))
    done()
    ro, rl = mo.mla_prefill_split(si.q_nope, si.q_pe, si.k_nope, si.k_pe, si.v, si.seq_len, 4, 2, si.scale, 1,
                                  prev_out=si.prev_out, prev_lse=si.prev_lse)
    assert_out_close(out, ro)
    assert_lse_close(lse, rl)


def step_cases(d):
    lens = [0, 10, 63, 64, 130]
    D = gen.decode_inputs([n + 1 for n in lens], H=16, seed=13, page_size=16)
    g = torch.Generator().manual_seed(14)
    B = len(lens)
    q_pe, c_kv, k_pe = gen.randn_bf16((B, 16, 64), g), gen.randn_bf16((B, 512), g), gen.randn_bf16((B, 64), g)
    pos = torch.tensor(lens, dtype=torch.int32)
    cs = gen.rope_cos_sin(512)
    cache, q_out = D.cache.to(d), D.q.to(d).clone()
    lib.mla_rope_append(q_pe.to(d), c_kv.to(d), k_pe.to(d), pos.to(d), cs.to(d), cache, D.block_table.to(d), q_out)
    done()
    q_rope, new_cache = mo.mla_rope_append(q_pe, c_kv, k_pe, pos, cs, False, D.cache, D.block_table, 16)
    assert_out_close(q_out[:, :, 512:], q_rope, tol=5e-2)
    assert_out_close(cache, new_cache, tol=5e-2)
    wk, wv = gen.absorb_weights(16, seed=15)
    qn = gen.randn_bf16((100, 16, 128), g)
    fused = torch.zeros((100, 16, 576), dtype=torch.bfloat16, device=d)
    lib.mla_absorb_q(qn.to(d), wk.to(d), q_out=fused)
    done()
    assert_out_close(fused[:, :, :512], mo.absorb_q(qn.double().numpy(), wk.double().numpy()), tol=5e-2)
    o = gen.randn_bf16((100, 16, 512), g)
    out = lib.mla_project_out(o.to(d), wv.to(d))
    done()
    assert_out_close(out, mo.project_out(o.double().numpy(), wv.double().numpy()), tol=5e-2)


if __name__ == "__main__":
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    for case in (prefill_cases, decode_cases, sparse_cases, split_merge_cases, step_cases):
        case(dev)
        print(case.__name__, "ok", flush=True)
    print("guarded ok")
