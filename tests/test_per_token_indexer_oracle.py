"""Oracle pins for per-token indexer keys.

Source: "V4 KV Layout: Classical + State dual pool": the State cache table keeps
one K-only indexer key per token, and a block holds 128 of them.  The pages do
not say how per-token scores rank CSA entries.  The reading taken here:
- An entry's score combines its m tokens' scores with the entry's indexer
  gates, s_e = sum_i sum_j alpha[j][i] <q_j, y_{m e + i, j}>.
- By linearity this is the per-entry score of the keys before the
  compressor's rounding.

The pins:
- Stored keys sit at their token's place.
- Scores follow the formula in float64 within fp32 rounding and agree with
  the per-entry variant.
- The top-k is taken over these scores.
- A prefix image (one run of keys per 32 tokens) restores bit for bit.
"""
import numpy as np
import pytest

import oracle as O
from heterogeneous_compressed_kv_gb300.gen import workloads as W
from tests import harness as H

TINY2 = dict(W.TINY, idx_heads=2, idx_dim=32, seed=61)  # two indexer heads: the gates mix per head


def _alpha(w, layer=0):
    """The oracle's gates: softmax in double, rounded to fp32."""
    g = H.gates(w)[2][layer].astype(np.float64)
    e = np.exp(g - g.max(axis=-1, keepdims=True))
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32).astype(np.float64)  # [Ih][m]


def _formula(w, y, qi, n_csa):
    """float64 s_e = sum_i sum_j alpha[j][i] <q_j, y_{4e+i, j}> and the
    matching magnitude bound sum |alpha| |q| |y|."""
    m, Ih, Id = w["m"], w["idx_heads"], w["idx_dim"]
    a = _alpha(w)
    yy = y[:n_csa * m].astype(np.float64).reshape(n_csa, m, Ih, Id)
    q = qi.astype(np.float64).reshape(Ih, Id)
    dots = np.einsum("emjd,jd->emj", yy, q)
    mags = np.einsum("emjd,jd->emj", np.abs(yy), np.abs(q))
    return np.einsum("emj,jm->e", dots, a), np.einsum("emj,jm->e", mags, np.abs(a))


def _filled(w, n_tokens, per_token=1):
    o = H.make_oracle(dict(w, idx_per_token=per_token), 2, 8, 6)
    r = o.alloc_request()[1]
    k, v, x = H.tokens(w, [0], [0], [n_tokens])
    assert o.append([r], [n_tokens], k, v, x) == 0
    return o, r, x[0]


@pytest.mark.parametrize("w", [dict(W.TINY, seed=60), TINY2], ids=["one_head", "two_heads"])
def test_scores_follow_the_formula_and_equal_the_per_entry_scores(w):
    n = 3 * 128 + 45  # three sealed blocks and a staged tail (including an open CSA group)
    o, r, y = _filled(w, n)
    oe, re_, _ = _filled(w, n, per_token=0)
    n_csa = n // w["m"]
    _, qi = H.queries(w, 0, [0], 0)
    rc, s = o.request_scores(0, r, qi[0], n_csa)
    rc2, s_entry = oe.request_scores(0, re_, qi[0], n_csa)
    assert rc == rc2 == 0
    ref, mag = _formula(w, y, qi[0], n_csa)
    bound = 2e-6 * mag + 1e-30  # a few fp32 roundings of terms bounded by mag
    assert np.all(np.abs(s - ref) <= bound), np.max(np.abs(s - ref) / bound)
    assert np.all(np.abs(s_entry - ref) <= bound)  # linearity: the same score up to rounding


def test_a_wrong_gate_index_is_caught_by_the_formula():
    """The pin has teeth: swapping the gates' head and token indices moves
    the scores far outside the bound."""
    w = TINY2
    n = 200
    o, r, y = _filled(w, n)
    n_csa = n // w["m"]
    _, qi = H.queries(w, 0, [0], 1)
    s = o.request_scores(0, r, qi[0], n_csa)[1]
    ref, mag = _formula(w, y, qi[0], n_csa)
    m, Ih, Id = w["m"], w["idx_heads"], w["idx_dim"]
    a = _alpha(w)
    yy = y[:n_csa * m].astype(np.float64).reshape(n_csa, m, Ih, Id)
    wrong = np.einsum("emjd,jd,mj->e", yy, qi[0].astype(np.float64).reshape(Ih, Id), a[:, :m].T[:, ::-1])
    assert np.max(np.abs(s - ref) / (mag + 1e-30)) < 1e-5
    assert np.max(np.abs(wrong - ref) / (mag + 1e-30)) > 1e-3


def test_stored_keys_are_the_tokens_own_keys():
    """fp32 cache: every token's key (sealed or staged) is stored exactly, at
    its position; bf16 cache: rounded to bf16."""
    import torch
    for w in (dict(W.TINY, seed=62), dict(W.TINY, in_dtype=W.BF16, cache_dtype=W.BF16, seed=63)):
        n = 2 * 128 + 7
        o, r, y = _filled(w, n)
        for t in list(range(0, n, 17)) + [127, 128, n - 1]:
            rc, code, _ = o.request_entry(0, r, 3, t)
            assert rc == 0
            if w["cache_dtype"] == W.F32:
                got = code.view(np.float32)
                assert np.array_equal(got, y[t].astype(np.float32)), t
            else:
                got = code.view(np.uint16).astype(np.uint32) << 16
                want = torch.from_numpy(y[t].astype(np.float32)).bfloat16().float().numpy()
                assert np.array_equal(got.view(np.float32), want), t
        assert o.request_entry(0, r, 3, n)[0] == O.ERR_INVALID_ARG  # past the last token


def test_decode_selects_the_top_k_of_these_scores():
    w = dict(TINY2, seed=64)
    n = 3 * 128 + 21
    o, r, _ = _filled(w, n)
    n_csa = n // w["m"]
    q, qi = H.queries(w, 0, [0], 2)
    rc, _, tk = o.decode_attend(0, [r], q, qi, 16)
    assert rc == 0
    s = o.request_scores(0, r, qi[0], n_csa)[1]
    assert np.array_equal(tk[0], O.topk(s, 16))


def test_prefix_image_holds_one_run_of_keys_per_32_tokens_and_restores():
    """fp8 keys: the block's indexer part is m runs of 32 keys (chunk-major
    codes, then 32 scales padded to 16 bytes); an image restores every key
    and score bit for bit; the per-token fingerprint differs from the
    per-entry one."""
    w = dict(W.TINY, in_dtype=W.BF16, cache_dtype=W.FP8, idx_heads=2, idx_dim=32, seed=65)
    n = 2 * 128
    o, r, _ = _filled(w, n)
    oe, _, _ = _filled(w, n, per_token=0)
    assert o.fingerprint() != oe.fingerprint()
    xsz, CB = 64, 32
    run = CB * xsz + 64  # 32 bf16 scales = 64 bytes, already a multiple of 16
    assert o.image_bytes(n, 0) - oe.image_bytes(n, 0) == 2 * (4 * run - run)
    rc, img = o.export_prefix(r, n, 0)
    assert rc == 0 and img.size == o.image_bytes(n, 0)
    r2 = o.alloc_request()[1]
    k, v, _ = H.tokens(w, [0], [n - w["n_win"]], [w["n_win"]])
    assert o.import_prefix(r2, img, k, v) == 0
    for t in range(0, n, 5):
        a, b = o.request_entry(0, r, 3, t), o.request_entry(0, r2, 3, t)
        assert a[0] == b[0] == 0 and np.array_equal(a[1], b[1]) and a[2][0] == b[2][0]
    _, qi = H.queries(w, 0, [0], 3)
    s1 = o.request_scores(0, r, qi[0], n // 4)[1]
    s2 = o.request_scores(0, r2, qi[0], n // 4)[1]
    assert np.array_equal(s1, s2)
