"""Every plausible mistake planted in a copy of the oracle is caught by a pin.

Each mutation rewrites one expression of oracle/oracle.c (a dropped term, a
wrong sign, index or operand), compiles the copy into a temporary library and
runs the pins of tests/oracle_pins.py against it; at least one pin must fail.
This shows the pins constrain the oracle, not just agree with it.  The real
oracle is never modified.  Each mutant runs in a child process, since a
broken index can also read past a host buffer; a crash counts as caught.
"""
import os
import subprocess
import sys

import pytest

import oracle
from tests import oracle_pins

MUTATIONS = [
    ("gqa-mapping-decode", "attend(&pv, qv, h / group,", "attend(&pv, qv, h % num_kv_heads,"),
    ("gqa-mapping-extend", "attend(&pv, q + at, h / group,", "attend(&pv, q + at, h % num_kv_heads,"),
    ("scale-dropped", "s *= scale;", "s *= 1.0;"),
    ("max-sign", "exp(scores[j - j0] - m)", "exp(m - scores[j - j0])"),
    ("no-normalise", "o[c] = o[c] / l;", "o[c] = o[c];"),
    ("lse-no-max", "*lse = m + log(l);", "*lse = log(l);"),
    ("causal-excludes-self", "cached_lens[r] + t + 1;", "cached_lens[r] + t;"),
    ("causal-sees-next", "cached_lens[r] + t + 1;", "cached_lens[r] + t + 2;"),
    ("extend-skips-first", "rows, 0, visible,", "rows, 1, visible,"),
    ("extend-packing", "tok += extend_lens[r];", "tok += cached_lens[r];"),
    ("v-from-k-pool", "pv->v_pool + (int64_t)rows[j]", "pv->k_pool + (int64_t)rows[j]"),
    ("v-logical-index", "(int64_t)rows[j] * pv->row_stride", "(int64_t)j * pv->row_stride"),
    ("k-head-offset-dropped", "row * pv->row_stride + (int64_t)kv_head * d;",
     "row * pv->row_stride;"),
    ("q-transposed", "*qv = q + ((int64_t)r * num_q_heads + h) * head_dim;",
     "*qv = q + ((int64_t)h * batch + r) * head_dim;"),
    ("decode-short-by-one", "j1 = j_end[r];", "j1 = j_end[r] - 1;"),
    ("widen-wrong-shift", "(uint32_t)bits << 16", "(uint32_t)bits << 15"),
    ("store-v-at-token-index", "memcpy(v_pool + row * pool_row_stride",
     "memcpy(v_pool + i * pool_row_stride"),
    ("store-k-gets-v", "memcpy(k_pool + row * pool_row_stride, k + i * tok_stride",
     "memcpy(k_pool + row * pool_row_stride, v + i * tok_stride"),
    ("merge-unweighted", "o[c] += w * os[c];", "o[c] += os[c];"),
    ("merge-lse-no-max", "lse_out[i] = top + log(total);", "lse_out[i] = log(total);"),
    ("rope-first-half-sign", "out[at + j] = x1 * c - x2 * s;", "out[at + j] = x1 * c + x2 * s;"),
    ("rope-second-half-sign", "out[at + half + j] = x2 * c + x1 * s;",
     "out[at + half + j] = x2 * c - x1 * s;"),
    ("rope-adjacent-pairs", "x2 = widen(x[at + half + j]);", "x2 = widen(x[at + (j ^ 1)]);"),
    ("rope-cos-sin-swapped", "const double c = (double)cs[j], s = (double)cs[half + j];",
     "const double s = (double)cs[j], c = (double)cs[half + j];"),
    ("rope-position-off-by-one", "cos_sin_cache + pos * head_dim;", "cos_sin_cache + (pos + 1) * head_dim;"),
    ("rope-heads-transposed", "const int64_t at = (i * num_heads + h) * (int64_t)head_dim;",
     "const int64_t at = (h * n_tokens + i) * (int64_t)head_dim;"),
    ("rope-no-range-check", "if (pos < 0 || pos >= max_positions)", "if (pos < 0)"),
    ("weights-skip-first", "for (int64_t j = j0; j < j1; j++) {\n        double w",
     "for (int64_t j = j0 + 1; j < j1; j++) {\n        double w"),
]


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = """
import sys
sys.path.insert(0, {root!r})
import oracle
from tests import oracle_pins
mut = oracle.Oracle({lib!r})
for pin in oracle_pins.ALL_PINS:
    try:
        pin(mut)
    except (AssertionError, ValueError):
        print('caught by', pin.__name__)
        sys.exit(0)
sys.exit(3)
"""


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutation site for {name} must be unique in oracle.c"
    mutant_src = tmp_path / "mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib = oracle.compile_oracle(str(mutant_src), str(tmp_path / "libmutant.so"))
    res = subprocess.run([sys.executable, "-c", _CHILD.format(root=ROOT, lib=lib)],
                         capture_output=True, text=True, timeout=300)
    # 0: a pin failed; negative: the mutant crashed the child; 3: it survived
    assert res.returncode != 3, f"mutation {name} survived every pin"
    assert res.returncode == 0 or res.returncode < 0, res.stderr[-2000:]
