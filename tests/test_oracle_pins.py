"""Pins for the CPU oracle: facts fixed by the pages and by mathematics.

Each check is a function of the oracle routine under test, so the mutation
tests at the end can plant a plausible mistake in a copy of the oracle (on the
CPU) and show that some pin catches it.
"""

from __future__ import annotations

import math
import os

import numpy as np
import pytest
import torch

from oracle import dcp_oracle as orc
import helpers as H

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# slot map
# ---------------------------------------------------------------------------

def check_slot_map_bijection(slot_map_fn, S, I, N, bs):
    sm = slot_map_fn([S], I, N, bs)
    shard = sm["shard_of"][0, :S]
    local = sm["local_pos"][0, :S]
    assert (shard >= 0).all() and (shard < N).all()
    for r in range(N):
        mine = np.nonzero(shard == r)[0]
        # local positions of shard r are exactly 0..n-1, increasing with t
        assert np.array_equal(local[mine], np.arange(len(mine)))
        assert sm["local_seq_lens"][r, 0] == len(mine)
        assert sm["local_num_blocks"][r, 0] == -(-len(mine) // bs)
    assert sm["local_seq_lens"][:, 0].sum() == S


def closed_form_local(t, I, N):
    return (t // (I * N)) * I + t % I


def closed_form_len(S, r, I, N):
    rem = S % (I * N) - r * I
    return (S // (I * N)) * I + min(max(rem, 0), I)


def check_slot_map_closed_form(slot_map_fn, S, I, N, bs):
    sm = slot_map_fn([S], I, N, bs)
    t = np.arange(S)
    assert np.array_equal(sm["local_pos"][0, :S], closed_form_local(t, I, N))
    for r in range(N):
        assert sm["local_seq_lens"][r, 0] == closed_form_len(S, r, I, N)


SLOT_CASES = [(1, 1, 1, 16), (1, 16, 2, 16), (17, 16, 2, 16), (1024, 16, 2, 16),
              (1000, 1, 8, 128), (129, 128, 4, 128), (5000, 128, 8, 128),
              (513, 7, 3, 5), (300, 1000, 4, 16), (200, 50, 4, 8)]


@pytest.mark.parametrize("S,I,N,bs", SLOT_CASES)
def test_slot_map_bijection(S, I, N, bs):
    check_slot_map_bijection(orc.ref_slot_map, S, I, N, bs)


@pytest.mark.parametrize("S,I,N,bs", SLOT_CASES)
def test_slot_map_closed_form(S, I, N, bs):
    check_slot_map_closed_form(orc.ref_slot_map, S, I, N, bs)


def read_golden_split():
    meta, rows = {}, []
    with open(os.path.join(GOLDEN, "dcp_blog_contiguous_split.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0].isdigit():
                rows.append(tuple(int(x) for x in parts))
            else:
                meta[parts[0]] = int(parts[1])
    return meta, rows


def check_blog_example(slot_map_fn):
    meta, rows = read_golden_split()
    S, N, I = meta["seq_len"], meta["dcp_size"], meta["interleave"]
    sm = slot_map_fn([S], I, N, 128)
    shard = sm["shard_of"][0]
    for r, lo, hi in rows:
        assert (shard[lo:hi] == r).all(), f"shard {r} should hold [{lo},{hi})"
        assert sm["local_seq_lens"][r, 0] == hi - lo


def test_slot_map_blog_worked_example():
    check_blog_example(orc.ref_slot_map)


def test_slot_map_interleave_at_least_seq_len_is_all_on_shard0():
    sm = orc.ref_slot_map([100, 64], 128, 4, 16)
    assert (sm["shard_of"][0, :100] == 0).all()
    assert list(sm["local_seq_lens"][:, 0]) == [100, 0, 0, 0]
    assert list(sm["local_seq_lens"][:, 1]) == [64, 0, 0, 0]


# ---------------------------------------------------------------------------
# unsharded attention
# ---------------------------------------------------------------------------

def rand(shape, seed, std=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * std


def check_vs_sdpa(attn_fn, B=2, Lq=3, Hq=8, Hkv=2, D=16, Dv=12, lens=(9, 31), scale=0.3):
    """Oracle vs torch SDPA (fp64, CPU) with an explicit causal-tail mask."""
    q = rand((B, Lq, Hq, D), 1)
    Ks = [rand((S, Hkv, D), 10 + b) for b, S in enumerate(lens)]
    Vs = [rand((S, Hkv, Dv), 20 + b) for b, S in enumerate(lens)]
    out, _ = attn_fn(q, Ks, Vs, np.array(lens), scale, Lq)
    g = Hq // Hkv
    for b, S in enumerate(lens):
        qt = torch.from_numpy(q[b]).permute(1, 0, 2)                      # [Hq][Lq][D]
        kt = torch.from_numpy(Ks[b]).permute(1, 0, 2).repeat_interleave(g, 0)  # [Hq][S][D]
        vt = torch.from_numpy(Vs[b]).permute(1, 0, 2).repeat_interleave(g, 0)
        i = torch.arange(Lq)[:, None]
        t = torch.arange(S)[None, :]
        mask = t <= (S - Lq + i)
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt, kt, vt, attn_mask=mask, scale=scale)                     # [Hq][Lq][Dv]
        err = np.abs(out[b] - ref.permute(1, 0, 2).numpy()).max()
        assert err < 1e-12, err


def test_attn_matches_torch_sdpa():
    check_vs_sdpa(orc.ref_attn_unsharded)


def test_attn_matches_torch_sdpa_mla_shape():
    check_vs_sdpa(orc.ref_attn_unsharded, B=1, Lq=4, Hq=16, Hkv=1, D=40, Dv=32, lens=(23,))


def check_brute_force(attn_fn):
    """n <= 8 keys: every exp and sum written out with math.exp / math.fsum."""
    Lq, Hq, Hkv, D = 1, 4, 2, 5
    for n in range(1, 9):
        q = rand((1, Lq, Hq, D), 100 + n)
        K = rand((n, Hkv, D), 200 + n)
        V = rand((n, Hkv, 3), 300 + n)
        scale = 0.7
        out, lse = attn_fn(q, [K], [V], np.array([n]), scale, Lq)
        for h in range(Hq):
            g = h // (Hq // Hkv)
            s = [scale * math.fsum(q[0, 0, h, d] * K[t, g, d] for d in range(D)) for t in range(n)]
            e = [math.exp(x) for x in s]
            tot = math.fsum(e)
            assert abs(lse[0, 0, h] - math.log(tot)) < 1e-12
            for d in range(3):
                ref = math.fsum(e[t] * V[t, g, d] for t in range(n)) / tot
                assert abs(out[0, 0, h, d] - ref) < 1e-12


def test_attn_brute_force_small():
    check_brute_force(orc.ref_attn_unsharded)


def test_attn_single_key_returns_value():
    q = rand((1, 1, 2, 6), 5)
    K = rand((1, 1, 6), 6)
    V = rand((1, 1, 4), 7)
    out, lse = orc.ref_attn_unsharded(q, [K], [V], np.array([1]), 0.5, 1)
    for h in range(2):
        assert np.allclose(out[0, 0, h], V[0, 0], atol=1e-15)
        assert abs(lse[0, 0, h] - 0.5 * float(q[0, 0, h] @ K[0, 0])) < 1e-12


def test_attn_constant_keys_give_mean_of_values():
    n = 37
    q = rand((1, 1, 3, 8), 8)
    k = rand((8,), 9)
    K = np.tile(k, (n, 1, 1))
    V = rand((n, 1, 5), 10)
    out, lse = orc.ref_attn_unsharded(q, [K], [V], np.array([n]), 0.25, 1)
    for h in range(3):
        assert np.allclose(out[0, 0, h], V[:, 0].mean(axis=0), atol=1e-13)
        assert abs(lse[0, 0, h] - (math.log(n) + 0.25 * float(q[0, 0, h] @ k))) < 1e-12


def check_causal(attn_fn):
    S, Lq = 20, 4
    q = rand((1, Lq, 2, 6), 11)
    K = rand((S, 1, 6), 12)
    V = rand((S, 1, 3), 13)
    out, lse = attn_fn(q, [K], [V], np.array([S]), 0.4, Lq)
    # the last query sees every key: same as a single query over all S keys
    o1, l1 = attn_fn(q[:, Lq - 1:], [K], [V], np.array([S]), 0.4, 1)
    assert np.allclose(out[0, Lq - 1], o1[0, 0], atol=1e-14)
    assert np.allclose(lse[0, Lq - 1], l1[0, 0], atol=1e-14)
    # query 0 sees S - Lq + 1 keys
    n0 = S - Lq + 1
    o0, l0 = attn_fn(q[:, :1], [K[:n0]], [V[:n0]], np.array([n0]), 0.4, 1)
    assert np.allclose(out[0, 0], o0[0, 0], atol=1e-14)
    assert np.allclose(lse[0, 0], l0[0, 0], atol=1e-14)


def test_attn_causal_tail():
    check_causal(orc.ref_attn_unsharded)


# ---------------------------------------------------------------------------
# shards + merge
# ---------------------------------------------------------------------------

def merged_vs_unsharded(w, decode_fn=None, attn_fn=None):
    inst = H.build_instance(w)
    res = (decode_fn or H.oracle_decode)(inst)
    q, _, _, sl = H.oracle_inputs(inst)
    Ks, Vs = H.logical_kv(inst)
    full, full_lse = (attn_fn or orc.ref_attn_unsharded)(q, Ks, Vs, sl, w.scale, w.q_len)
    out = orc.head_slices(full, w.dcp_size)
    out_lse = orc.head_slices(full_lse, w.dcp_size)
    return res, out, out_lse


MERGE_CASES = [
    ("tiny_gqa", dict(lengths=("fixed", 77))),
    ("tiny_gqa", dict(lengths=("fixed", 77), dcp_size=4, interleave=1)),
    ("tiny_gqa", dict(lengths=("fixed", 200), dcp_size=8, interleave=5, block_size=4)),
    ("tiny_gqa", dict(lengths=("fixed", 50), dcp_size=4, interleave=64)),   # empty shards
    ("tiny_gqa", dict(batch=3, q_len=3, lengths=("uniform", 3, 90), dcp_size=2, interleave=7)),
    ("mla_mtp", dict(num_q_heads=8, head_dim_qk=40, head_dim_v=32, lengths=("fixed", 150),
                     dcp_size=4, interleave=1, block_size=16)),
    ("mla_32", dict(batch=2, num_q_heads=8, head_dim_qk=24, head_dim_v=16,
                    lengths=("uniform", 60, 300), dcp_size=8, interleave=16, block_size=16)),
]


@pytest.mark.parametrize("name,kw", MERGE_CASES)
def test_merge_equals_unsharded(name, kw):
    w = H.small(name, **kw)
    res, out, out_lse = merged_vs_unsharded(w)
    assert np.abs(res["out"] - out).max() < 1e-12
    assert np.abs(res["out_lse"] - out_lse).max() < 1e-12


@pytest.mark.parametrize("N", [1, 2, 4, 8])
def test_merge_invariant_in_dcp_size(N):
    base = H.small("mla_32", batch=2, num_q_heads=8, head_dim_qk=24, head_dim_v=16,
                   lengths=("uniform", 100, 400), interleave=8, block_size=8)
    inst1 = H.build_instance(base.with_(dcp_size=1))
    ref = H.oracle_decode(inst1)
    got = H.oracle_decode(H.repage(inst1, base.with_(dcp_size=N)))
    full_ref = ref["out"][0]
    full_got = np.concatenate(list(got["out"]), axis=2)   # undo the head slicing
    assert np.abs(full_ref - full_got).max() < 1e-12
    lse_ref = ref["out_lse"][0]
    lse_got = np.concatenate(list(got["out_lse"]), axis=2)
    assert np.abs(lse_ref - lse_got).max() < 1e-12


def test_merge_n1_is_identity():
    rng = np.random.default_rng(3)
    p = rng.standard_normal((1, 2, 1, 4, 5))
    l = rng.standard_normal((1, 2, 1, 4))
    out, out_lse = orc.ref_merge(p, l)
    assert np.allclose(out, p, atol=1e-15) and np.allclose(out_lse, l, atol=1e-15)


def test_merge_two_shards_closed_form():
    a, b = 0.3, -1.7
    o1, o2 = np.array([1.0, -2.0]), np.array([0.5, 4.0])
    p = np.stack([o1, o2])[:, None, None, None, :]       # [2][1][1][1][2]
    p = np.repeat(p, 2, axis=3)                          # Hq = 2 so Hq % N == 0
    l = np.array([a, b])[:, None, None, None].repeat(2, axis=3)
    out, out_lse = orc.ref_merge(p, l)
    ea, eb = math.exp(a), math.exp(b)
    assert abs(out_lse[0, 0, 0, 0] - math.log(ea + eb)) < 1e-14
    assert np.allclose(out[0, 0, 0, 0], (ea * o1 + eb * o2) / (ea + eb), atol=1e-14)


def test_merge_all_empty_gives_zero_and_neg_inf():
    p = np.zeros((2, 1, 1, 2, 3))
    l = np.full((2, 1, 1, 2), -np.inf)
    out, out_lse = orc.ref_merge(p, l)
    assert (out == 0).all() and (out_lse == -np.inf).all()


def test_empty_shard_partial():
    w = H.small("tiny_gqa", lengths=("fixed", 20), dcp_size=4, interleave=32)
    res = H.oracle_decode(H.build_instance(w))
    assert (res["lse"][1:] == -np.inf).all()
    assert (res["partial_out"][1:] == 0).all()
    assert np.isfinite(res["lse"][0]).all()


def test_head_slice_enumeration():
    rng = np.random.default_rng(4)
    full = rng.standard_normal((2, 3, 8, 5))
    sl = orc.head_slices(full, 4)
    for r in range(4):
        for hp in range(2):
            assert np.array_equal(sl[r, :, :, hp], full[:, :, r * 2 + hp])


# ---------------------------------------------------------------------------
# planted mistakes: each must be caught by at least one pin above
# ---------------------------------------------------------------------------

def _wrong_shard_slot_map(seq_lens, I, N, bs):
    """Plausible mistake: rotate the owner by one shard."""
    sm = orc.ref_slot_map(seq_lens, I, N, bs)
    shard = sm["shard_of"]
    shard[shard >= 0] = (shard[shard >= 0] + 1) % N
    sm["local_seq_lens"] = np.roll(sm["local_seq_lens"], 1, axis=0)
    sm["local_num_blocks"] = np.roll(sm["local_num_blocks"], 1, axis=0)
    return sm


def _wrong_local_order_slot_map(seq_lens, I, N, bs):
    """Plausible mistake: shard-local order reversed."""
    sm = orc.ref_slot_map(seq_lens, I, N, bs)
    for b, S in enumerate(seq_lens):
        for r in range(N):
            idx = np.nonzero(sm["shard_of"][b, :S] == r)[0]
            sm["local_pos"][b, idx] = sm["local_pos"][b, idx][::-1]
    return sm


def _attn_with(mistake):
    def fn(q, keys, values, seq_lens, scale, q_len):
        q = np.asarray(q, dtype=np.float64)
        B, Lq, Hq, _ = q.shape
        Hkv = keys[0].shape[1]
        Dv = values[0].shape[2]
        out = np.zeros((B, Lq, Hq, Dv))
        lse = np.zeros((B, Lq, Hq))
        for b in range(B):
            S = int(seq_lens[b])
            for i in range(Lq):
                last = S - Lq + i + (1 if mistake == "causal_off_by_one" else 0)
                last = min(last, S - 1)
                for h in range(Hq):
                    g = h % Hkv if mistake == "kv_head_mod" else h // (Hq // Hkv)
                    k = keys[b][: last + 1, g]
                    v = values[b][: last + 1, g]
                    sc = 1.0 if mistake == "no_scale" else scale
                    s = sc * (k @ q[b, i, h])
                    m = s.max()
                    p = np.exp(s - m)
                    if mistake == "lse_without_max":
                        out[b, i, h] = (p @ v) / p.sum()
                        lse[b, i, h] = math.log(p.sum())
                    else:
                        out[b, i, h] = (p @ v) / p.sum()
                        lse[b, i, h] = m + math.log(p.sum())
        return out, lse
    return fn


def _caught(check, *args):
    try:
        check(*args)
    except AssertionError:
        return True
    return False


def test_planted_slot_map_mistakes_are_caught():
    assert _caught(check_blog_example, _wrong_shard_slot_map)
    assert _caught(check_slot_map_closed_form, _wrong_local_order_slot_map, 1000, 16, 4, 16)
    assert _caught(check_slot_map_bijection, _wrong_local_order_slot_map, 1000, 16, 4, 16)


@pytest.mark.parametrize("mistake", ["causal_off_by_one", "kv_head_mod", "no_scale",
                                     "lse_without_max"])
def test_planted_attention_mistakes_are_caught(mistake):
    fn = _attn_with(mistake)
    caught = (_caught(check_vs_sdpa, fn) or _caught(check_brute_force, fn)
              or _caught(check_causal, fn))
    assert caught, mistake
    # and the correct oracle passes the same checks
    check_vs_sdpa(orc.ref_attn_unsharded)
    check_brute_force(orc.ref_attn_unsharded)
    check_causal(orc.ref_attn_unsharded)


def test_planted_merge_mistake_is_caught():
    """A merge that forgets to normalise by sum_r exp(lse_r) breaks the invariance pin."""
    def bad_merge(partial_out, lse):
        N = partial_out.shape[0]
        w = np.exp(lse)[..., None]
        full = (w * partial_out).sum(axis=0)
        return orc.head_slices(full, N), orc.head_slices(np.log(np.exp(lse).sum(axis=0)), N)

    w = H.small("tiny_gqa", lengths=("fixed", 60), dcp_size=2, interleave=4)
    inst = H.build_instance(w)
    q, kv, bt, sl = H.oracle_inputs(inst)
    parts = [orc.ref_attn_shard("gqa", q, kv, bt, sl, r, 2, 4, w.block_size, w.scale, 1, 64)
             for r in range(2)]
    out_bad, _ = bad_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    _, out, _ = merged_vs_unsharded(w)
    assert np.abs(out_bad - out).max() > 1e-6
