"""The CPU oracle against its pins, and the pins against planted mistakes."""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
import oracle_pins

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


@pytest.mark.parametrize("pin", oracle_pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle.load())


def test_kv_cache_count():
    oracle_pins.pin_kv_cache_count()


# Each mutant plants one plausible mistake in a copy of the oracle's C source.
# Every mutant must make at least one pin fail.
MUTANTS = {
    "pool_scale_dropped": ("s[t] = scale * acc / (double)r;", "s[t] = acc / (double)r;"),
    "pool_sum_not_mean_over_heads": ("s[t] = scale * acc / (double)r;", "s[t] = scale * acc;"),
    "pool_first_token_query": ("const int64_t last = (j + 1) * g - 1;", "const int64_t last = j * g;"),
    "pool_not_normalised": ("const double a = s[t] / den;", "const double a = s[t];"),
    "pool_values_weighted_by_keys": ("vc[c] += a * v[c];", "vc[c] += a * k[c];"),
    "partial_group_visible": ("const int64_t n_core = window_lo(i, w) / g;",
                              "const int64_t n_core = (window_lo(i, w) + g - 1) / g;"),
    "one_core_too_few": ("const int64_t n_core = window_lo(i, w) / g;",
                         "const int64_t n_core = window_lo(i, w) / g > 0 ? window_lo(i, w) / g - 1 : 0;"),
    "aligned_window_not_aligned": ("const int64_t lo = window_mode ? n_core * g : window_lo(i, w);",
                                   "const int64_t lo = window_lo(i, w);"),
    "max_pool_takes_min": ("km = kv_ > km ? kv_ : km;", "km = kv_ < km ? kv_ : km;"),
    "mean_pool_not_uniform": ("for (int64_t t = 0; t < g; ++t) s[t] = 0.0; /* mean pooling: equal weights */",
                              "(void)0; /* mean pooling: equal weights */"),
    "window_too_wide": ("return i - w + 1 > 0 ? i - w + 1 : 0;", "return i - w > 0 ? i - w : 0;"),
    "window_too_narrow": ("return i - w + 1 > 0 ? i - w + 1 : 0;", "return i - w + 2 > 0 ? (i - w + 2 < i ? i - w + 2 : i) : 0;"),
    "core_scale_dropped": ("z[j] = scale * dot;", "z[j] = dot;"),
    "local_scale_dropped": ("z[n_core + m] = scale * dot;", "z[n_core + m] = dot;"),
    "lse_log2": ("*lse = mx + log(den);", "*lse = mx + log2(den);"),
    "core_output_uses_keys": ("o[c] += a * Vch[j * d + c];", "o[c] += a * Kch[j * d + c];"),
    "local_keys_reversed": ("dot += q[c] * Kh[(lo + m) * d + c];", "dot += q[c] * Kh[(i - m) * d + c];"),
    "core_logit_uses_values": ("dot += q[c] * Kch[j * d + c];", "dot += q[c] * Vch[j * d + c];"),
    "gqa_post_mean_no_1_over_r": ("wsum[t] += exp(s[t] - hmx) / hden / (double)r;",
                                  "wsum[t] += exp(s[t] - hmx) / hden;"),
    "gqa_post_mean_not_normalised_per_head": ("wsum[t] += exp(s[t] - hmx) / hden / (double)r;",
                                              "wsum[t] += exp(s[t] - hmx) / (double)r;"),
    "gqa_post_mean_is_logit_mean": ("if (pool_mode == 3) {", "if (pool_mode == 99) {"),
    "gqa_post_mean_first_head_only": ("wsum[t] += exp(s[t] - hmx) / hden / (double)r;\n                }",
                                      "wsum[t] += exp(s[t] - hmx) / hden / (double)r;\n                    break;\n                }"),
    "gqa_post_mean_values_weighted_by_keys": ("vc[c] += wsum[t] * v[c];", "vc[c] += wsum[t] * k[c];"),
    "gqa_post_mean_head_scale_dropped": ("s[t] = scale * dot;\n                    }\n                    double hmx",
                                         "s[t] = dot;\n                    }\n                    double hmx"),
    "kv_head_interleaved": ("const int64_t bk = b * Hkv + h / r;\n            attend_row(Q + u * d",
                            "const int64_t bk = b * Hkv + h % Hkv;\n            attend_row(Q + u * d"),
}


@pytest.fixture(scope="module")
def mutant_dir():
    d = tempfile.mkdtemp(prefix="cca_oracle_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, mutant_dir):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "cca_oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    msrc = os.path.join(mutant_dir, name + ".c")
    with open(msrc, "w") as f:
        f.write(src.replace(old, new, 1))
    so = oracle.build(force=True, src=msrc, out=os.path.join(mutant_dir, name + ".so"))
    lib = oracle.load(so)
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin caught mutant {name}"


@pytest.mark.parametrize("pin", oracle_pins.BACKWARD_PINS, ids=lambda f: f.__name__)
def test_backward_pin(pin):
    pin(oracle.load())


def test_backward_forward_matches_c_oracle():
    """The differentiable dense forward of the backward oracle equals the C oracle."""
    import numpy as np
    import torch
    from oracle.backward import dense_forward
    rng = np.random.default_rng(70)
    Q, K, V = (rng.standard_normal(s) for s in ((2, 4, 32, 8), (2, 2, 32, 8), (2, 2, 32, 8)))
    for g, w, pm, wm in ((4, 5, 0, 0), (8, 9, 1, 1), (2, 3, 2, 0), (4, 6, 3, 0), (2, 5, 3, 1)):
        O, L = dense_forward(torch.tensor(Q), torch.tensor(K), torch.tensor(V), g, w, pool_mode=pm, window_mode=wm)
        Or, Lr, _, _ = oracle.prefill(Q, K, V, g, w, pool_mode=pm, window_mode=wm)
        np.testing.assert_allclose(O.numpy(), Or, rtol=0, atol=1e-12)
        np.testing.assert_allclose(L.numpy(), Lr, rtol=0, atol=1e-12)
