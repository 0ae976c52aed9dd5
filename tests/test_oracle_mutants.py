"""Plant plausible mistakes in a copy of the oracle and check the pins catch each.

Every mutant is oracle.c with one substring replaced, compiled into a temporary
directory and run against the full pin battery in a child process (a mutant
that crashes counts as caught as well).  The real oracle is untouched.
"""
import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "head_group_modulo": ("const int kv = h / G;", "const int kv = h % Hkv;"),
    "slot_reversed": ("int64_t slot = tok % block_size;",
                      "int64_t slot = (block_size - 1) - tok % block_size;"),
    "scale_dropped": ("s[t] = scale * dot;", "s[t] = dot;"),
    "max_is_min": ("if (s[t] > m) m = s[t];", "if (s[t] < m) m = s[t];"),
    "not_normalised": ("out[d] /= z;", "out[d] /= 1.0;"),
    "exp_sign": ("s[t] = exp(s[t] - m);", "s[t] = exp(m - s[t]);"),
    "exp_base_two": ("s[t] = exp(s[t] - m);", "s[t] = exp2(s[t] - m);"),
    "values_from_k": ("out[d] += s[t] * (vs[t] * load_elem(v_pool,",
                      "out[d] += s[t] * (vs[t] * load_elem(k_pool,"),
    "e4m3_bias": ("ldexp(1.0 + (double)m / 8.0, e - 7)", "ldexp(1.0 + (double)m / 8.0, e - 8)"),
    "e4m3_subnormal": ("ldexp((double)m / 8.0, -6)", "ldexp((double)m / 8.0, -7)"),
    "e4m3_sign_lost": ("return sign ? -x : x;", "return x;"),
    "k_scale_ignored": ("ks[t] = k_scale ? (double)k_scale[sc_idx] : 1.0;", "ks[t] = 1.0;"),
    "v_scale_ignored": ("vs[t] = v_scale ? (double)v_scale[sc_idx] : 1.0;", "vs[t] = 1.0;"),
    "v_scale_from_k_table": ("vs[t] = v_scale ? (double)v_scale[sc_idx] : 1.0;",
                             "vs[t] = v_scale ? (double)k_scale[sc_idx] : 1.0;"),
    "block_scale_by_logical_block": (
        "const int64_t sc_idx = scale_per_block ? phys * Hkv + kv : kv;",
        "const int64_t sc_idx = scale_per_block ? (tok / block_size) * Hkv + kv : kv;"),
    "block_scale_head_dropped": ("const int64_t sc_idx = scale_per_block ? phys * Hkv + kv : kv;",
                                 "const int64_t sc_idx = scale_per_block ? phys * Hkv : kv;"),
    "block_scale_ignored": ("const int64_t sc_idx = scale_per_block ? phys * Hkv + kv : kv;",
                            "const int64_t sc_idx = kv;"),
    "int8_read_unsigned": ("return (double)((const int8_t *)base)[idx];",
                           "return (double)((const uint8_t *)base)[idx];"),
    "query_head_index": ("* Hq + h) * (int64_t)D", "* Hq + kv) * (int64_t)D"),
    "query_token_index": ("((int64_t)b * q_len + i) * Hq", "((int64_t)b * q_len) * Hq"),
    "causal_shifted": ("const int64_t p = L - q_len + i;", "const int64_t p = L - q_len + i - 1;"),
    "window_off_by_one": ("if (window > 0 && p - window + 1 > 0) lo = p - window + 1;",
                          "if (window > 0 && p - window > 0) lo = p - window;"),
    "window_ignored": ("if (window > 0 && p - window + 1 > 0) lo = p - window + 1;", ""),
    "bf16_shift": ("<< 16;", "<< 15;"),
    "pool_axes_swapped": ("((phys * block_size + slot) * Hkv + kv)",
                          "((phys * Hkv + kv) * block_size + slot)"),
    "length_off_by_one": ("const int64_t L = seq_lens[b];",
                          "const int64_t L = seq_lens[b] > 1 ? seq_lens[b] - 1 : seq_lens[b];"),
}

RUNNER = textwrap.dedent("""
    import sys
    sys.path.insert(0, {root!r})
    sys.path.insert(0, {tests!r})
    import oracle
    from oracle_pins import PINS
    orc = oracle.Oracle({lib!r})
    failed = []
    for pin in PINS:
        try:
            pin(orc)
        except Exception as e:
            failed.append(pin.__name__)
    print("FAILED:" + ",".join(failed))
    sys.exit(1 if failed else 0)
""")


def _build_mutant(tmp_path, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site must be unique: %r" % old
    path = tmp_path / "oracle_mutant.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", str(path), "-o", str(lib),
                    "-lm"], check=True, capture_output=True)
    return str(lib)


def _run_pins(lib):
    code = RUNNER.format(root=ROOT, tests=os.path.join(ROOT, "tests"), lib=lib)
    return subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                          timeout=300)


def test_unmutated_copy_passes(tmp_path):
    lib = _build_mutant(tmp_path, "const int kv = h / G;", "const int kv = h / G;")
    res = _run_pins(lib)
    assert res.returncode == 0, res.stdout + res.stderr


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    old, new = MUTANTS[name]
    lib = _build_mutant(tmp_path, old, new)
    res = _run_pins(lib)
    assert res.returncode != 0, "mutant %s survived every pin" % name
