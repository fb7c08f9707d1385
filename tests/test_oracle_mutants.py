"""The oracle's pins have teeth: each plausible mistake planted in a copy of the
oracle (on the CPU, never in the CUDA path) makes at least one pin test fail.

Each mutant is a textual change of the oracle's C source, compiled into a
temporary library and loaded by a child pytest run of tests/test_oracle_pins.py
through the ZERO_ORACLE_LIB variable.
"""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle")

# (name, file, original text, mutated text)
MUTANTS = [
    ("sum_not_mean", "zero_oracle.c", "return g * inv_n;", "return g;"),
    ("m_sign", "zero_oracle.c", "s->b1 * *m + s->omb1 * g", "s->b1 * *m - s->omb1 * g"),
    ("v_linear_in_g", "zero_oracle.c", "s->omb2 * g * g", "s->omb2 * g"),
    ("bias_correction_index", "zero_oracle.c", "pow(hp->beta1, t)", "pow(hp->beta1, t + 1.0)"),
    ("eps_inside_sqrt", "zero_oracle.c", "sqrtf(vh) + s->eps", "sqrtf(vh + s->eps)"),
    ("no_weight_decay", "zero_oracle.c", "+ s->wd * w0)", "+ 0.0f * w0)"),
    ("lr_sign", "zero_oracle.c", "float w1 = w0 - s->lr", "float w1 = w0 + s->lr"),
    ("betas_swapped", "zero_oracle.c", "s->b1 = (float)hp->beta1;", "s->b1 = (float)hp->beta2;"),
    ("floor_padding", "zero_oracle.c", "if (n_chunks * chunk < p)\n            n_chunks += 1;", ""),
    ("params_from_m", "zero_oracle.c", "params_bf16[i] = or_bf16_rne(master[k][j]);",
     "params_bf16[i] = or_bf16_rne(m[k][j]);"),
    ("zero2_grads_unsharded", "zero_oracle.c", "out->grad_bytes = stage >= 2", "out->grad_bytes = stage >= 3"),
    ("zero3_volume_2P", "zero_oracle.c", "stage == 3 ? 3.0 * P : 2.0 * P", "2.0 * P"),
    ("bf16_ties_up", "zero_oracle.c", "keep = (below & 1u) ? below + 1u : below;", "keep = below + 1u;"),
    ("gather_ignores_unit_offset", "zero_oracle.c", "shard_bf16[k][unit->shard_offset + j];",
     "shard_bf16[k][j];"),
    ("reverse_rank_order", "zero_oracle.c",
     "for (int32_t r = 0; r < n_ranks; ++r)\n        g = g + or_bf16_to_f32(grads[r][i]);",
     "for (int32_t r = n_ranks - 1; r >= 0; --r)\n        g = g + or_bf16_to_f32(grads[r][i]);"),
    ("clip_coef_from_sumsq", "zero_oracle.c", "double norm = sqrt(sumsq);", "double norm = sumsq;"),
    ("clip_not_clamped", "zero_oracle.c", "    if (c > 1.0)\n        c = 1.0;\n", ""),
    ("clip_eps_dropped", "zero_oracle.c", "double c = max_norm / (norm + 1e-6);",
     "double c = max_norm / norm;"),
    ("clip_coef_unused", "zero_oracle.c", "float g = or_reduce_mean(grads, n_ranks, i, s.inv_n) * coef;",
     "float g = or_reduce_mean(grads, n_ranks, i, s.inv_n);"),
    ("accumulator_restarts", "zero_oracle.c", "float a = first ? 0.0f : grad_acc[k][j];",
     "float a = 0.0f;"),
    ("accumulation_not_averaged", "zero_oracle.c",
     "float g = (a + or_reduce_mean(grads, n_ranks, i, s.inv_n)) * inv_m;",
     "float g = (a + or_reduce_mean(grads, n_ranks, i, s.inv_n));"),
    ("zero2_accum_volume_mP", "zero_oracle.c", "case 2: return m * P + P;", "case 2: return m * P;"),
    ("f32_mean_not_scaled", "zero_oracle.c",
     "        g = g + grads[r][i];\n    return g * inv_n;", "        g = g + grads[r][i];\n    return g;"),
    ("generator_lane_dropped", "gen_oracle.c", "(int32_t)(h >> 48) - 131070", "(int32_t)(h >> 48) * 0 - 131070"),
    ("reshard_source_rank_from_new_layout", "zero_oracle.c",
     "x = src[i / from->shard_len][from->shard_offset + i % from->shard_len];",
     "x = src[i / to->shard_len % n_from][from->shard_offset + i % from->shard_len];"),
    ("reshard_ignores_unit_offset", "zero_oracle.c", "dst[k][to->shard_offset + j] = x;",
     "dst[k][j] = x;"),
    ("sampled_clip_first_coef_every_step", "zero_oracle.c", "g = g * coef[t];",
     "g = g * coef[0];"),
    ("sampled_clip_coef_ignored", "zero_oracle.c", "g = g * coef[t];", "g = g * 1.0f;"),
    ("sampled_accum_one_short", "zero_oracle.c",
     "for (int32_t mu = 1; mu < micro_batches - 1; ++mu)",
     "for (int32_t mu = 2; mu < micro_batches - 1; ++mu)"),
    ("sampled_accum_not_averaged", "zero_oracle.c", "g = (a + g) * inv_m;", "g = (a + g);"),
]


def _build_mutant(tmp, fname, old, new):
    for f in ("zero_oracle.c", "gen_oracle.c", "zero_oracle.h"):
        text = open(os.path.join(SRC, f)).read()
        if f == fname:
            assert old in text, "mutation target vanished from %s: %r" % (f, old)
            text = text.replace(old, new, 1)
        open(os.path.join(tmp, f), "w").write(text)
    lib = os.path.join(tmp, "liboracle_mutant.so")
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-std=c11", "-shared", "-fPIC", "-o", lib,
                    os.path.join(tmp, "zero_oracle.c"), os.path.join(tmp, "gen_oracle.c"), "-lm"],
                   check=True)
    return lib


def _run_mutant(mutant):
    """Builds one mutant and runs the pins against it: (pytest's exit code, the
    end of its output), or (None, the error) if the mutant could not be built."""
    name, fname, old, new = mutant
    try:
        with tempfile.TemporaryDirectory() as tmp:
            lib = _build_mutant(tmp, fname, old, new)
            env = dict(os.environ, ZERO_ORACLE_LIB=lib)
            r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p",
                                "no:cacheprovider",
                                os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                               cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
            return r.returncode, r.stdout[-2000:]
    except Exception as e:  # reported by the mutant's own test
        return None, repr(e)


@pytest.fixture(scope="module")
def mutant_runs():
    """Every mutant built and run against the pins, as many at a time as the
    host has cores (each run is a separate process and library)."""
    import concurrent.futures as cf
    workers = max(1, min(len(MUTANTS), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        return dict(zip([m[0] for m in MUTANTS], ex.map(_run_mutant, MUTANTS)))


@pytest.mark.parametrize("name,fname,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(mutant_runs, name, fname, old, new):
    code, out = mutant_runs[name]
    assert code == 1, "mutant %s survived the pins (exit %s):\n%s" % (name, code, out)
