"""The attention parity bounds have teeth (CPU only).

At the long-context shape ("Why does V4 split pools? ..." s4: one softmax
over [selected CSA entries | every HCA entry | the SWA window]; 2,048 + 8,192
+ 128 sources, fp8 e4m3 cache with bf16 scales, 16 heads x 128) the output is
an average over ~10^4 sources and its entries are of order 1e-2.  These tests
check, on the oracle's own output, that the bounds the GPU parity tests apply
(tests.gpu_harness.check_out) reject outputs that are wrong: all zeros, a
source class missing, or a single source missing; and that the max-abs bound
alone would not.

Sources: K and V values drawn per head from a normal distribution with the
spread of the workload's compressed entries (a softmax-gated sum of m
N(0, 1) tokens has standard deviation sqrt(sum_i alpha_i^2) per head), window
tokens N(0, 1); every source is encoded to the fp8 cache format by the
oracle.
"""
import numpy as np
import pytest

import oracle as O
from heterogeneous_compressed_kv_gb300 import kvpool as K
from heterogeneous_compressed_kv_gb300.gen import workloads as W
from tests import harness as H
from tests.gpu_harness import check_out, tol


@pytest.fixture(scope="module")
def long_context_sources():
    w = dict(W.LONG_CONTEXT)
    heads, hd = w["heads"], w["head_dim"]
    g_csa, g_hca, _ = H.gates(w)
    sig_csa = np.sqrt([(O.softmax_f32(g_csa[0][h]).astype(np.float64) ** 2).sum() for h in range(heads)])
    sig_hca = np.sqrt([(O.softmax_f32(g_hca[0][h]).astype(np.float64) ** 2).sum() for h in range(heads)])
    o = H.make_oracle(w, 1, 1, 1)
    rng = np.random.default_rng(2024)

    def entries(n, sig):
        codes = np.empty((n, o.esz), np.uint8)
        scales = np.empty((n, 2), np.uint16)
        for j in range(n):
            k = (rng.standard_normal((heads, hd)) * sig[:, None]).reshape(-1)
            v = (rng.standard_normal((heads, hd)) * sig[:, None]).reshape(-1)
            ck, sk = O.encode(w["cache_dtype"], k)
            cv, sv = O.encode(w["cache_dtype"], v)
            codes[j] = np.concatenate([ck, cv])
            scales[j] = (sk, sv)
        return codes, scales

    src = {"csa": entries(w["top_k"], sig_csa),
           "hca": entries(w["length"] // w["m_prime"], sig_hca),
           "win": entries(w["n_win"], np.ones(heads))}
    q = rng.standard_normal(heads * hd).astype(np.float32)

    def attend(drop=(), cut=None):
        """The oracle's output over the sources, without the classes in
        `drop` and, if cut = (class, j), without source j of that class."""
        cs, ss = [], []
        for name in ("csa", "hca", "win"):
            if name in drop:
                continue
            c, s = src[name]
            if cut is not None and cut[0] == name:
                keep = np.arange(len(c)) != cut[1]
                c, s = c[keep], s[keep]
            cs.append(c)
            ss.append(s)
        rc, out = o.attend_sources(np.concatenate(cs), np.concatenate(ss), q)
        assert rc == 0
        return out

    return w, attend, attend()


def test_fp8_bounds_accept_the_reference(long_context_sources):
    w, _, ref = long_context_sources
    assert w["cache_dtype"] == K.FP8_E4M3
    err, rel = check_out(ref, ref, w["cache_dtype"])
    assert err == 0.0 and rel == 0.0


def test_fp8_max_abs_alone_has_no_teeth(long_context_sources):
    # why the rel-L2 bound is needed: an all-zero output is within max-abs
    w, _, ref = long_context_sources
    amax, rl2 = tol(w["cache_dtype"])
    assert np.abs(ref).max() < amax
    assert rl2 is not None


@pytest.mark.parametrize("wrong", ["zeros", "no_window", "no_hca", "no_csa", "half_hca", "one_window_token_less",
                                   "one_csa_entry_less"])
def test_fp8_bounds_reject_wrong_outputs(long_context_sources, wrong):
    w, attend, ref = long_context_sources
    bad = {"zeros": lambda: np.zeros_like(ref),
           "no_window": lambda: attend(drop=("win",)),
           "no_hca": lambda: attend(drop=("hca",)),
           "no_csa": lambda: attend(drop=("csa",)),
           "half_hca": lambda: 0.5 * (attend(drop=("hca",)) + ref),
           "one_window_token_less": lambda: attend(cut=("win", 0)),
           "one_csa_entry_less": lambda: attend(cut=("csa", 7))}[wrong]()
    with pytest.raises(AssertionError, match=r"(rel-L2|max-abs) error"):
        check_out(bad, ref, w["cache_dtype"])


def test_fp8_bounds_accept_the_expected_gpu_error(long_context_sources):
    # each weight p * V-scale rounded to f16 (the GPU's largest own error
    # source): perturb every source's weight by a relative 2^-11 at most, which
    # moves the output by about 2.8e-4 rel-L2, inside the bound
    w, _, ref = long_context_sources
    rng = np.random.default_rng(7)
    noisy = ref * (1.0 + rng.uniform(-2.0 ** -11, 2.0 ** -11, ref.shape))
    check_out(noisy, ref, w["cache_dtype"])
