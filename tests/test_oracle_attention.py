"""Pins for the oracle's attention and for the whole oracle decode step.

What fixes the answer: with every page selected the result is ordinary
softmax attention, which torch's scaled_dot_product_attention computes
independently (in fp64 on the CPU); the SequenceO1 close reading (§5.1)
gives exactly this debugging check (100% retention must equal full
attention).  Split-and-merge by log-sum-exp must give the union's result
(the reduction of split rows, SALS AICPU Tiling challenge 2); the result
cannot depend on where pages sit in the physical pool; a single token gives
its own value row.
"""

import math

import numpy as np
import pytest
import torch

from oracle import attention, decode


def _sdpa(q, k, v, scale):
    qt = torch.from_numpy(q)[None, None]
    kt = torch.from_numpy(k)[None, None]
    vt = torch.from_numpy(v)[None, None]
    return torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)[0, 0].numpy()


def test_attend_matches_library_sdpa(rng):
    for trial in range(10):
        G, T, d = int(rng.integers(1, 9)), int(rng.integers(1, 300)), 64
        q = rng.standard_normal((G, d))
        k = rng.standard_normal((T, d)) * 2
        v = rng.standard_normal((T, d))
        out, lse = attention.attend(q, k, v, 1 / math.sqrt(d))
        ref = _sdpa(q, k, v, 1 / math.sqrt(d))
        assert np.abs(out - ref).max() < 1e-12
        z = q @ k.T / math.sqrt(d)
        assert np.allclose(lse, np.log(np.exp(z).sum(axis=1)), rtol=1e-12)


def test_single_token(rng):
    q = rng.standard_normal((2, 16))
    k = rng.standard_normal((1, 16))
    v = rng.standard_normal((1, 16))
    out, lse = attention.attend(q, k, v, 0.25)
    assert np.allclose(out, np.repeat(v, 2, axis=0), rtol=0, atol=1e-15)
    assert np.allclose(lse, (q @ k.T)[:, 0] * 0.25, rtol=1e-14)


def test_empty_token_set():
    out, lse = attention.attend(np.ones((3, 8)), np.zeros((0, 8)), np.zeros((0, 8)), 1.0)
    assert (out == 0).all() and np.isneginf(lse).all()


def test_lse_combine_of_splits_equals_union(rng):
    G, T, d = 4, 257, 32
    q = rng.standard_normal((G, d))
    k = rng.standard_normal((T, d))
    v = rng.standard_normal((T, d))
    whole = attention.attend(q, k, v, 0.3)
    for n_split in (1, 2, 3, 7, 16):
        cuts = np.linspace(0, T, n_split + 1).astype(int)
        parts = [attention.attend(q, k[a:b], v[a:b], 0.3) for a, b in zip(cuts[:-1], cuts[1:])]
        parts.append(attention.attend(q, k[:0], v[:0], 0.3))  # an empty split
        out, lse = attention.lse_combine(parts)
        assert np.abs(out - whole[0]).max() < 1e-12
        assert np.abs(lse - whole[1]).max() < 1e-12


def _tiny_inputs(rng, lens, S=4, Hkv=2, G=2, d=8, int8=False, perm=True):
    pages = [-(-L // S) for L in lens]
    n_phys = sum(pages)
    order = rng.permutation(n_phys) if perm else np.arange(n_phys)
    pt = np.full((len(lens), max(pages + [1])), -1)
    off = 0
    for b in range(len(lens)):
        pt[b, : pages[b]] = order[off : off + pages[b]]
        off += pages[b]
    if int8:
        kp = rng.integers(-127, 128, (n_phys, Hkv, S, d)).astype(np.int8)
        vp = rng.integers(-127, 128, (n_phys, Hkv, S, d)).astype(np.int8)
        ks = (rng.random((n_phys, Hkv, S)) * 0.05 + 0.01).astype(np.float16)
        vs = (rng.random((n_phys, Hkv, S)) * 0.05 + 0.01).astype(np.float16)
    else:
        kp = rng.standard_normal((n_phys, Hkv, S, d)).astype(np.float16)
        vp = rng.standard_normal((n_phys, Hkv, S, d)).astype(np.float16)
        ks = vs = None
    q = rng.standard_normal((len(lens), Hkv * G, d)).astype(np.float16)
    return decode.StepInputs(q, kp, vp, ks, vs, pt, np.array(lens))


def _dense_reference(inp, b, h, S):
    """Brute force: walk logical tokens 0..L-1 through the page table."""
    L = int(inp.seq_lens[b])
    G = inp.group
    ks, vs = [], []
    for t in range(L):
        phys = inp.page_table[b][t // S]
        k = inp.k_pool[phys, h, t % S].astype(np.float64)
        v = inp.v_pool[phys, h, t % S].astype(np.float64)
        if inp.k_scale is not None:
            k = k * float(inp.k_scale[phys, h, t % S])
            v = v * float(inp.v_scale[phys, h, t % S])
        ks.append(k)
        vs.append(v)
    q = inp.q[b, h * G : (h + 1) * G].astype(np.float64)
    if not ks:
        return np.zeros_like(q), np.full(G, -np.inf)
    k, v = np.array(ks), np.array(vs)
    d = q.shape[1]
    out = _sdpa(q, k, v, 1 / math.sqrt(d))
    lse = np.log(np.exp(q @ k.T / math.sqrt(d)).sum(axis=1))
    return out, lse


@pytest.mark.parametrize("int8", [False, True])
def test_all_pages_selected_equals_dense(rng, int8):
    S = 4
    inp = _tiny_inputs(rng, [13, 4, 1, 0, 9], S=S, int8=int8)
    for selector in ("quest", "all"):
        prm = decode.StepParams(page_size=S, n_sel=64, n_sink=1, n_recent=1, selector=selector, head_dim=8)
        if selector == "quest" and int8:
            continue
        res = decode.decode_step(inp, prm)
        for (b, h), out in res["out"].items():
            ref_out, ref_lse = _dense_reference(inp, b, h, S)
            assert np.abs(out - ref_out).max() < 1e-12
            assert np.allclose(res["lse"][(b, h)], ref_lse, rtol=1e-12) or np.isneginf(ref_lse).all()


def test_physical_placement_does_not_matter(rng):
    S = 4
    inp = _tiny_inputs(rng, [23, 11], S=S, perm=False)
    prm = decode.StepParams(page_size=S, n_sel=3, n_sink=1, n_recent=1, selector="quest", head_dim=8)
    base = decode.decode_step(inp, prm)
    perm = rng.permutation(inp.k_pool.shape[0])
    inv = np.argsort(perm)
    moved = decode.StepInputs(
        inp.q, inp.k_pool[perm], inp.v_pool[perm], None, None,
        np.where(inp.page_table >= 0, inv[np.maximum(inp.page_table, 0)], -1), inp.seq_lens,
    )
    res = decode.decode_step(moved, prm)
    assert res["sel"] == base["sel"]
    for key in base["out"]:
        assert np.array_equal(res["out"][key], base["out"][key])


def test_tokens_past_seq_len_are_ignored(rng):
    S = 4
    inp = _tiny_inputs(rng, [10], S=S)
    prm = decode.StepParams(page_size=S, n_sel=2, n_sink=1, n_recent=1, selector="quest", head_dim=8)
    base = decode.decode_step(inp, prm)
    phys = inp.page_table[0][2]
    inp.k_pool[phys, :, 2:] = 50
    inp.v_pool[phys, :, 2:] = 50
    res = decode.decode_step(inp, prm)
    assert res["sel"] == base["sel"]
    for key in base["out"]:
        assert np.array_equal(res["out"][key], base["out"][key])


def test_planted_mistake_is_caught(rng, monkeypatch):
    """Dropping the softmax scale must fail the library comparison."""
    real = attention.attend
    monkeypatch.setattr(attention, "attend", lambda q, k, v, scale: real(q, k, v, 1.0))
    with pytest.raises(AssertionError):
        test_attend_matches_library_sdpa(rng)
