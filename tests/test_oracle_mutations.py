"""The oracle's pins catch plausible mistakes (CPU).

Each case plants one mistake in a copy of oracle/pa_oracle.c -- a wrong GQA
head map, a causal limit off by one, a wrong slot inside a page, a dropped
score scale, a sink with the wrong sign, values read from the key cache, a
split partial whose max is not in the log2 domain, a reduce that forgets the
exp-sum weights, a scatter into the wrong slot or of padding tokens, and in
the quantised cache a wrong E4M3 exponent bias, ties rounded to odd, a wrong
quantisation or stored scale, padding tokens quantised -- rebuilds that copy in
a temporary tree and runs the pins (tests/test_oracle_pins.py,
tests/test_oracle_fp8.py) against it: at least one pin must fail.  The
repository's own oracle is not touched.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, exact line fragment of pa_oracle.c, planted replacement)
MUTATIONS = [
    ("gqa_head_map",
     "const int g = h / (a->num_q_heads / a->num_kv_heads);",
     "const int g = h % a->num_kv_heads;"),
    ("causal_off_by_one",
     "if (a->causal && N - n + i < last) last = N - n + i;",
     "if (a->causal && N - n + i - 1 < last) last = N - n + i - 1;"),
    ("slot_inside_page",
     "int64_t slot = (int64_t)page * a->block_size + j % a->block_size;",
     "int64_t slot = (int64_t)page * a->block_size + (j + 1) % a->block_size;"),
    ("dropped_scale",
     "s_buf[j] = a->scale * dot;",
     "s_buf[j] = dot;"),
    ("sink_sign",
     "if (a->sinks) den += exp(sink - m);",
     "if (a->sinks) den += exp(-sink - m);"),
    ("values_from_key_cache",
     "for (int d = 0; d < D; ++d) o[d] += p * elem(a->value_cache, vo + d, a->kv_dtype);",
     "for (int d = 0; d < D; ++d) o[d] += p * elem(a->key_cache, vo + d, a->kv_dtype);"),
    ("partial_max_natural_units",
     "double t2 = scale * dot * log2e;",
     "double t2 = scale * dot;"),
    ("reduce_weight",
     "double w = PART(part_l, slot) * exp2(PART(part_m, slot) - M);",
     "double w = exp2(PART(part_m, slot) - M);"),
    ("scatter_slot",
     "int64_t page = slot / block_size, off = slot % block_size;",
     "int64_t page = slot / block_size, off = (slot + 1) % block_size;"),
    ("scatter_padding",
     "if (slot < 0) continue; /* padding token */\n        if (slot >= num_blocks * block_size) return -1;\n        int64_t page",
     "if (slot < 0) slot = 0;\n        if (slot >= num_blocks * block_size) return -1;\n        int64_t page"),
    # the quantised cache (pins in tests/test_oracle_fp8.py)
    ("e4m3_exponent_bias",
     "else v = ldexp(1.0 + (double)m / 8.0, e - 7);",
     "else v = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("e4m3_ties_to_odd",
     "best = (elo < ehi || (elo == ehi && (lo & 1) == 0)) ? lo : hi;",
     "best = (elo < ehi || (elo == ehi && (lo & 1) == 1)) ? lo : hi;"),
    ("quantise_inverse_scale",
     "const float inv = 448.0f / amax;",
     "const float inv = 256.0f / amax;"),
    ("quantise_stored_scale",
     "scales[slot * num_kv_heads + h] = amax / 448.0f;",
     "scales[slot * num_kv_heads + h] = amax / 256.0f;"),
    ("quantise_padding",
     "if (slot < 0) continue; /* padding token */\n        if (slot >= num_blocks * block_size) return -1;\n        for (int which",
     "if (slot < 0) slot = 0;\n        if (slot >= num_blocks * block_size) return -1;\n        for (int which"),
]


def _tree(dst):
    """The files the pins need, copied under dst."""
    os.makedirs(os.path.join(dst, "oracle"))
    for f in ("__init__.py", "oracle.py"):
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(dst, "oracle", f))
    os.makedirs(os.path.join(dst, "paged_kv_varlen_gb300"))
    for f in ("__init__.py", "workloads.py"):
        shutil.copy(os.path.join(ROOT, "paged_kv_varlen_gb300", f),
                    os.path.join(dst, "paged_kv_varlen_gb300", f))
    os.makedirs(os.path.join(dst, "tests"))
    for f in ("conftest.py", "test_oracle_pins.py", "test_oracle_fp8.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))


def _run_pins(tree):
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    return subprocess.run(
        [sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
         os.path.join("tests", "test_oracle_pins.py"), os.path.join("tests", "test_oracle_fp8.py")],
        cwd=tree, env=env, capture_output=True, text=True, timeout=600)


def test_unmodified_copy_passes_its_pins(tmp_path):
    """The copied tree itself is sound: with the oracle unchanged every pin passes."""
    tree = str(tmp_path / "tree")
    _tree(tree)
    shutil.copy(os.path.join(ROOT, "oracle", "pa_oracle.c"), os.path.join(tree, "oracle"))
    res = _run_pins(tree)
    assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-2000:]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(tmp_path, name, old, new):
    src = open(os.path.join(ROOT, "oracle", "pa_oracle.c")).read()
    assert src.count(old) == 1, f"{name}: the line to mutate is not unique in pa_oracle.c"
    tree = str(tmp_path / "tree")
    _tree(tree)
    with open(os.path.join(tree, "oracle", "pa_oracle.c"), "w") as fh:
        fh.write(src.replace(old, new))
    res = _run_pins(tree)
    assert res.returncode == 1 and " failed" in res.stdout, (
        f"{name} survived the pins:\n" + res.stdout[-2000:] + res.stderr[-2000:])
