"""Prefix caching end to end on the GPU.

Request A writes its 40-token prompt (P 16) and caches its two full blocks;
request B shares A's first 32 tokens, starts from those cached blocks
(gk_seq_create_cached) and writes only its own 9 tokens.  Both attend a HOT
system prefix that the first acquire writes and the second finds cached
(gk_prefix_acquire).  A token's K/V depend only on its id and position, so B's
attention over the reused blocks must equal the fp64 oracle over B's own
context, for both backends."""
import numpy as np
import pytest

from oracle import attention
from parity import assert_attention_close
from synth.gen import KIND_PREFIX_K, KIND_PREFIX_V, KIND_SUFFIX_K, KIND_SUFFIX_V, bf16_bits_to_f64, normal_bits, stream_key

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from paged_kv_cache_pool_gb300 import binding as gk  # noqa: E402

HQ, HKV, D, P = 8, 2, 128, 16


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_pool_gb300 import build
    build.build()


def _kv_bits(kind, token, pos):
    return normal_bits(stream_key(41, kind, token, pos), 0, HKV * D).reshape(HKV, D)


def _rows(kind, tokens, pos0=0):
    return np.stack([_kv_bits(kind, t, pos0 + i) for i, t in enumerate(tokens)])   # [n, Hkv, d] bf16 bits


def _dev(bits):
    return torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).cuda()


def test_cached_blocks_and_hot_slab_decode_like_fresh_ones():
    from paged_kv_cache_pool_gb300.engine import Engine
    rng = np.random.default_rng(5)
    eng = Engine(1, HQ, HKV, D, 512, 64 * P, P, seed=3)
    try:
        pool = eng.pool
        sys_tokens = rng.integers(0, 30000, 100).tolist()
        a_tokens = rng.integers(0, 30000, 40).tolist()
        b_tokens = a_tokens[:32] + rng.integers(0, 30000, 9).tolist()

        # HOT system prefix: written once, found cached the second time
        base, hit = gk.gk_prefix_acquire(pool, 0xABCDEF, len(sys_tokens))
        assert not hit
        eng.write_prefix(0, base, len(sys_tokens), 0, _dev(_rows(KIND_PREFIX_K, sys_tokens)),
                         _dev(_rows(KIND_PREFIX_V, sys_tokens)))
        base2, hit2 = gk.gk_prefix_acquire(pool, 0xABCDEF, len(sys_tokens))
        assert hit2 and base2 == base

        # COLD: A writes everything and caches its full blocks; B reuses them
        seqs = []
        for toks in (a_tokens, b_tokens):
            sid, n_cached = gk.gk_seq_create_cached(pool, toks)
            seqs.append(sid)
            rest = toks[n_cached:]
            slots, cow = eng.append_slots(np.full(len(rest), sid, dtype=np.int32))
            assert len(cow) == 0
            eng.append_kv(0, eng.to_device(slots), _dev(_rows(KIND_SUFFIX_K, rest, n_cached)),
                          _dev(_rows(KIND_SUFFIX_V, rest, n_cached)))
            gk.gk_seq_cache_blocks(pool, sid, toks)
            if toks is b_tokens:
                assert n_cached == 32
        ta, _ = gk.gk_seq_table(pool, seqs[0])
        tb, _ = gk.gk_seq_table(pool, seqs[1])
        assert tb[:2].tolist() == ta[:2].tolist()          # B reads A's blocks

        table = eng.block_tables(seqs)
        d_table = eng.to_device(table)
        b = eng.batch([base, base], [len(sys_tokens)] * 2, [len(a_tokens), len(b_tokens)], d_table, table.shape[1])
        qbits = normal_bits(stream_key(41, 99), 0, 2 * HQ * D).reshape(2, HQ, D)
        q = _dev(qbits)
        plan = eng.plan(b)
        for backend in (gk.GK_BACKEND_CASCADE, gk.GK_BACKEND_DENSE):
            out = torch.empty((2, HQ, D), dtype=torch.float32, device="cuda")
            lse = torch.empty((2, HQ), dtype=torch.float32, device="cuda")
            b.set_device(d_q=q, d_out=out, d_lse=lse)
            eng.decode(0, b, plan, backend)
            torch.cuda.synchronize()
            assert eng.device_error() == gk.GK_OK
            for r, toks in enumerate((a_tokens, b_tokens)):
                k = np.concatenate([_rows(KIND_PREFIX_K, sys_tokens), _rows(KIND_SUFFIX_K, toks)])
                v = np.concatenate([_rows(KIND_PREFIX_V, sys_tokens), _rows(KIND_SUFFIX_V, toks)])
                o_ref, l_ref = attention.attend_heads(bf16_bits_to_f64(qbits[r]),
                                                      bf16_bits_to_f64(k).transpose(1, 0, 2),
                                                      bf16_bits_to_f64(v).transpose(1, 0, 2))
                assert_attention_close(out[r:r + 1].cpu().numpy(), lse[r:r + 1].cpu().numpy(),
                                       o_ref[None], l_ref[None], f"request {r} backend {backend}")
        gk.gk_prefix_unref(pool, 0xABCDEF)
        gk.gk_prefix_unref(pool, 0xABCDEF)
        assert gk.gk_hot_cache_stats(pool) == (1, 1, len(sys_tokens))
    finally:
        eng.close()
