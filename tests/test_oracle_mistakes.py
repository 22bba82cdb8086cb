"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (a dropped term, a wrong
index, sign, bias or offset), builds it with the same gcc flags into ``oracle/_variants/``
(git-ignored), swaps it in for the real oracle and runs the pins of ``test_oracle.py``: at
least one must fail. Every planted mistake keeps all memory accesses in bounds. This runs
on the CPU only; nothing here touches the CUDA library."""
import os
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle as pins

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "mla_oracle.c")
OUT = os.path.join(os.path.dirname(HERE), "oracle", "_variants")

# (name, exact text in mla_oracle.c, replacement)
MISTAKES = [
    ("causal window one key short", "int n = P->causal ? L - P->s_q + 1 + t : L;",
     "int n = P->causal ? L - P->s_q + t : L;"),
    ("RoPE term dropped", "w[(size_t)i * n + (j - lo)] = P->scale * (latent + rope);",
     "w[(size_t)i * n + (j - lo)] = P->scale * latent;"),
    ("scale not applied", "w[(size_t)i * n + (j - lo)] = P->scale * (latent + rope);",
     "w[(size_t)i * n + (j - lo)] = latent + rope;"),
    ("RoPE query against latent dims", "for (int r = 0; r < d_r; ++r) rope += qr[r] * key[d_c + r];",
     "for (int r = 0; r < d_r; ++r) rope += qr[r] * key[r];"),
    ("LSE without the row max", "lse[i] = m + log(l);", "lse[i] = log(l);"),
    ("LSE in base 2", "lse[i] = m + log(l);", "lse[i] = m + log2(l);"),
    ("weights not normalised", "for (int j = 0; j < n; ++j) s[j] = exp(s[j] - m) / l;",
     "for (int j = 0; j < n; ++j) s[j] = exp(s[j] - m);"),
    ("value read from shifted dims", "for (int d = 0; d < d_c; ++d) o[d] += p * key[d];",
     "for (int d = 0; d < d_c; ++d) o[d] += p * key[d + d_r];"),
    ("in-page offset and page index swapped", "return (int64_t)page * P->page_size + j % P->page_size;",
     "return (int64_t)page * P->page_size + j / P->page_size;"),
    ("query row ignores the new-token index", "int64_t qi = (((int64_t)b * P->s_q + t) * P->num_heads + heads[i]);",
     "int64_t qi = (((int64_t)b * P->s_q) * P->num_heads + heads[i]);"),
    ("E4M3 exponent bias 8", "v = ldexp(1.0 + (double)m / 8.0, e - 7);", "v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("E4M3 subnormal exponent", "v = ldexp((double)m / 8.0, -6);", "v = ldexp((double)m / 8.0, -7);"),
    ("E4M3 sign dropped", "return sign ? -v : v;", "return v;"),
    ("FP8 tile scale of the wrong tile", "memcpy(&sc, scales + 4 * (d / 128), sizeof sc);",
     "memcpy(&sc, scales + 4 * (d % 4), sizeof sc);"),
    ("merge weight inverted", "double wgt = exp(lses[i] - *lse);", "double wgt = exp(*lse - lses[i]);"),
    ("merge LSE without the max", "*lse = M + log(S);", "*lse = log(S);"),
]

PINS = [
    ("brute force", lambda: [pins.test_brute_force_tiny(s) for s in range(6)]),
    ("split == unsplit", lambda: [pins.test_split_merge_equals_unsplit(s) for s in range(5)]),
    ("absorb == expand", lambda: pins.test_absorb_equals_expand(4, 8, 4, 8, 16, 6, 6, 4)),
    ("weights sum to one", pins.test_weights_sum_to_one),
    ("uniform weights", pins.test_zero_query_gives_uniform_weights),
    ("single key", pins.test_single_key),
    ("dominant key", pins.test_dominant_key),
    ("duplicated keys", pins.test_duplicated_keys_add_ln2),
    ("page permutation", pins.test_page_permutation_invariance),
    ("E4M3 codes", pins.test_e4m3_all_codes_against_torch_and_definition),
    ("FP8 cache", pins.test_fp8_cache_matches_f64_cache),
]


def _build_variant(name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"anchor for '{name}' not found once in the oracle source"
    os.makedirs(OUT, exist_ok=True)
    tag = "".join(c if c.isalnum() else "_" for c in name)
    c_path, so_path = os.path.join(OUT, tag + ".c"), os.path.join(OUT, tag + ".so")
    with open(c_path, "w") as f:
        f.write(src.replace(old, new))
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", so_path, c_path, "-lm"])
    return so_path


def test_the_real_oracle_passes_every_pin():
    for _, pin in PINS:
        pin()


@pytest.mark.parametrize("name,old,new", MISTAKES, ids=[m[0] for m in MISTAKES])
def test_a_planted_mistake_fails_a_pin(name, old, new, monkeypatch):
    monkeypatch.setattr(oracle, "_lib", oracle.bind(_build_variant(name, old, new)))
    failed = []
    with np.errstate(all="ignore"):
        for pin_name, pin in PINS:
            try:
                pin()
            except AssertionError:
                failed.append(pin_name)
    assert failed, f"'{name}' passed every pin"
