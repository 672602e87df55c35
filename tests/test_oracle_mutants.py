"""The oracle's pins must catch plausible mistakes.

Each mutant below is a copy of the oracle source with one deliberate slip
planted in it (on the CPU, in a temporary directory).  The pin suite is run
against every mutant in a child process and must fail for each of them.
"""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "etc_oracle.cpp")

# (name, text in the source, replacement)
MUTANTS = [
    ("router_drops_bias", "if (bias) s += static_cast<double>(bias[e]);\n      logits[t * E + e] = s;",
     "logits[t * E + e] = s;"),
    ("router_transposed_weight", "bf16_to_double(wg[static_cast<long>(h) * E + e]);\n      if (bias) s",
     "bf16_to_double(wg[static_cast<long>(e) * H + h]);\n      if (bias) s"),
    ("ties_to_higher_id", "static_cast<double>(L[e]) > static_cast<double>(L[best])",
     "static_cast<double>(L[e]) >= static_cast<double>(L[best])"),
    ("weights_not_normalised", "w[j] = std::exp(static_cast<double>(L[ids[j]]) - l0) / z;",
     "w[j] = std::exp(static_cast<double>(L[ids[j]]) - l0);"),
    ("silu_wrong_sign", "act[n] = g / (1.0 + std::exp(-g)) * u;",
     "act[n] = g / (1.0 + std::exp(g)) * u;"),
    ("gate_up_swapped", "const uint16_t* wg_row = wgu_e + static_cast<long>(n) * H;",
     "const uint16_t* wg_row = wgu_e + static_cast<long>(I + n) * H;"),
    ("down_transposed", "const uint16_t* wd_row = wd_e + static_cast<long>(m) * I;\n    for (int n = 0; n < I; ++n) s += act[n] * bf16_to_double(wd_row[n]);",
     "for (int n = 0; n < I; ++n) s += act[n] * bf16_to_double(wd_e[static_cast<long>(n) * H + m]);"),
    ("unstable_permutation", "const long r = exp_indptr[e] + seen[e]++;",
     "const long r = exp_indptr[e + 1] - 1 - seen[e]++;"),
    ("combine_unweighted", "s += w[t * k + j] * y[static_cast<long>(pos[t * k + j]) * H + m];",
     "s += y[static_cast<long>(pos[t * k + j]) * H + m];"),
    ("mlp_ignores_row_list", "const long t = rows ? static_cast<long>(rows[i]) : i;",
     "const long t = i;"),
    ("splitk_drops_last_column", "for (long col = j * tile; col < (j + 1) * tile; ++col)",
     "for (long col = j * tile; col < (j + 1) * tile - 1; ++col)"),
    ("rmsnorm_sum_not_mean", "const double inv = 1.0 / std::sqrt(ss / H + eps);",
     "const double inv = 1.0 / std::sqrt(ss + eps);"),
    ("chain_drops_residual", "for (long i = 0; i < T * H; ++i) cur[i] += delta[i];",
     "for (long i = 0; i < T * H; ++i) cur[i] = delta[i];"),
    ("event_sim_ignores_wait", "if (counter[ev] == 0 && !final_queued[ev]) {",
     "if (!final_queued[ev]) {"),
]


def _run_mutant(name, old, new, tmp):
    import oracle
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutant {name}: anchor not found exactly once"
    path = os.path.join(tmp, f"{name}.cpp")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.oracle.compile_source(path, os.path.join(tmp, f"lib{name}.so"))
    env = dict(os.environ, ETC_ORACLE_LIB=lib, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-400:]


def test_every_mutant_is_caught():
    with tempfile.TemporaryDirectory() as tmp:
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            results = list(ex.map(lambda m: _run_mutant(*m, tmp), MUTANTS))
    survivors = [(n, out) for n, rc, out in results if rc == 0]
    assert not survivors, f"pins did not catch: {survivors}"
    # a failing pin run is a test failure (rc 1), not a crash or a usage error
    assert all(rc == 1 for _, rc, _ in results), results


def test_unmutated_source_passes():
    # Sanity check for the harness: the real oracle passes the pins when loaded
    # through the same ETC_ORACLE_LIB route.
    import oracle
    with tempfile.TemporaryDirectory() as tmp:
        lib = oracle.oracle.compile_source(SRC, os.path.join(tmp, "libsame.so"))
        env = dict(os.environ, ETC_ORACLE_LIB=lib)
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                            os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
