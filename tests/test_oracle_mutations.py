"""Mutation check of the oracle's pins (CPU only).

Each case plants one plausible mistake in a fresh copy of the oracle package
(its C file or its Python module), then runs the pins against that copy in a
child pytest process.  The conftest hook reads the PHOTON_ORACLE_UNDER_TEST
variable and imports the copy as ``oracle``.  Every mutant must make at least
one pin fail.  The unmutated copy must pass them all, which shows that the
copying itself changes nothing.

The mistakes are the ones a restatement of the pages' method could plausibly
contain:
* attention (README "Key features / GPU-optimized kernels": batched paged
  attention with a numerically stable softmax): the head map, the block-table
  walk, the scale, the max subtraction, the normaliser, the merge weights;
* the byte moves (README "Technical details / Paged attention": the batched
  cache write and the per-sequence block tables);
* the fp16 / bf16 / e4m3 decoders and the e4m3 encoder, the fp8 scales (README
  "Roadmap": lower-precision KV);
* RoPE (README "Key features / GPU-optimized kernels": batched RoPE);
* the scheduler's policy (README "Technical details / Continuous batching
  scheduler").
None of the mistakes makes the copy read or write outside its buffers.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_DIR = os.path.join(ROOT, "oracle")
PINS = ["tests/test_oracle_pins.py"]
SCHED_PINS = ["tests/test_scheduler_cpu.py", "-k", "golden_trace and oracle or oracle_invariants"]

C, PY, SCHED = "paged_ref.c", "__init__.py", "scheduler.py"

# (id, file, text to replace (must occur exactly once), replacement, pins)
MUTANTS = [
    # --- decode (C)
    ("kvh_map_modulo", C, "const int32_t kvh = h / G;", "const int32_t kvh = h % P->Hkv;", PINS),
    ("row_reversed_in_block", C, "+ kvh) * P->bs) + j % P->bs) * P->d;",
     "+ kvh) * P->bs) + (P->bs - 1 - j % P->bs)) * P->d;", PINS),
    ("table_entry_rotated", C, "int32_t blk = P->block_tables[(size_t)b * P->MBS + j / P->bs];",
     "int32_t blk = P->block_tables[(size_t)b * P->MBS + (j / P->bs + 1) % "
     "((P->context_lens[b] + P->bs - 1) / P->bs)];", PINS),
    ("scale_dropped", C, "s[j - j0] = P->scale * dot;", "s[j - j0] = dot;", PINS),
    ("max_not_subtracted", C, "double p = exp(s[j - j0] - m);", "double p = exp(s[j - j0]);",
     PINS),
    ("min_instead_of_max", C, "if (s[j - j0] > m) m = s[j - j0];",
     "if (j == j0 || s[j - j0] < m) m = s[j - j0];", PINS),
    ("first_key_dropped", C, "double p = exp(s[j - j0] - m);",
     "double p = (j == j0) ? 0.0 : exp(s[j - j0] - m);", PINS),
    ("k_used_as_v", C, "o[i] += p * load(P->v_cache,", "o[i] += p * load(P->k_cache,", PINS),
    ("normaliser_is_length", C, "for (int32_t i = 0; i < P->d; ++i) out[i] /= l;",
     "for (int32_t i = 0; i < P->d; ++i) out[i] /= (double)ctx;", PINS),
    ("merge_unweighted", C, "double w = exp(m[p] - M);", "double w = 1.0;", PINS),
    ("merge_denominator_unweighted", C, "den += w * l[p];", "den += l[p];", PINS),
    ("fp16_exponent_bias", C, "v = ldexp((double)(man | 0x400), ex - 25);",
     "v = ldexp((double)(man | 0x400), ex - 24);", PINS),
    ("fp16_subnormal_scale", C, "v = ldexp((double)man, -24);", "v = ldexp((double)man, -25);",
     PINS),
    ("bf16_shift", C, "uint32_t bits = (uint32_t)h << 16;", "uint32_t bits = (uint32_t)h << 15;",
     PINS),
    # --- byte moves (C)
    ("slot_offset_off_by_one", C, "int64_t blk = s / block_size, off = s % block_size;",
     "int64_t blk = s / block_size, off = (s + 1) % block_size;", PINS),
    ("gather_v_from_k_pool", C,
     "memcpy((char*)v_dense + dst, (const char*)v_cache + src, row);",
     "memcpy((char*)v_dense + dst, (const char*)k_cache + src, row);", PINS),
    ("cache_write_v_into_k_pool", C,
     "memcpy((char*)v_cache + dst, (const char*)v_new + src, row);",
     "memcpy((char*)v_cache + dst, (const char*)k_new + src, row);", PINS),
    # --- RoPE (C)
    ("rope_sign", C, "y[k] = a * c - b * s;", "y[k] = a * c + b * s;", PINS),
    ("rope_exponent", C, "pow(base, -2.0 * (double)k / (double)head_dim)",
     "pow(base, -(double)k / (double)head_dim)", PINS),
    ("rope_pairing", C, "const double a = x[k], b = x[k + half];",
     "const double a = x[k], b = x[(k + 1) % half + half];", PINS),
    # --- Python module: rounding, RoPE step, multi-query
    ("bf16_narrow_truncates", PY, "(b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))",
     "(b + np.uint32(0))", PINS),
    ("rope_step_position", PY, "pos = max(int(wl.context_lens[b]) - 1, 0)",
     "pos = int(wl.context_lens[b])", PINS),
    ("multi_query_own_key_dropped", PY, "rows_ctx.append(first + i + 1)",
     "rows_ctx.append(first + i)", PINS),
    # --- fp8 (Python module)
    ("e4m3_exponent_bias", PY, "np.power(2.0, e - 7)", "np.power(2.0, e - 8)", PINS),
    ("e4m3_subnormal_step", PY, "np.where(e == 0, m * 2.0 ** -9,", "np.where(e == 0, m * 2.0 ** -10,",
     PINS),
    ("e4m3_mantissa_sixteenths", PY, "(1.0 + m / 8.0)", "(1.0 + m / 16.0)", PINS),
    ("e4m3_ties_to_odd", PY, "((hi - a == a - lo) & (i % 2 == 0))",
     "((hi - a == a - lo) & (i % 2 == 1))", PINS),
    ("e4m3_overflow_to_nan", PY, "code = np.where(a >= _E4M3_POS[-1], 0x7E, code)",
     "code = np.where(a > _E4M3_POS[-1], 0x7F, code)", PINS),
    ("e4m3_sign_dropped", PY, "code = code.astype(np.int64) | np.where(np.signbit(v), 0x80, 0)",
     "code = code.astype(np.int64)", PINS),
    ("fp8_write_scale_not_inverted", PY, "inv = np.float32(1.0) / np.float32(scale)",
     "inv = np.float32(scale)", PINS),
    ("fp8_write_v_with_k_scale", PY, "(v_new, v_cache8, v_scale)", "(v_new, v_cache8, k_scale)",
     PINS),
    ("fp8_write_pools_swapped", PY,
     "((k_new, k_cache8, k_scale), (v_new, v_cache8, v_scale))",
     "((k_new, v_cache8, k_scale), (v_new, k_cache8, v_scale))", PINS),
    ("fp8_write_row_off_by_one", PY, "dst[slot // bs, :, slot % bs, :] = e4m3_encode(x)",
     "dst[slot // bs, :, (slot + 1) % bs, :] = e4m3_encode(x)", PINS),
    ("fp8_decode_v_scale_dropped", PY, "return out * float(v_scale)", "return out", PINS),
    ("fp8_decode_k_scale_dropped", PY, "float(scale) * float(k_scale),", "float(scale),", PINS),
    # --- scheduler (Python)
    ("sched_free_list_lifo", SCHED, "r.table.append(self.free.pop(0))",
     "r.table.append(self.free.pop())", SCHED_PINS),
    ("sched_preempt_oldest", SCHED, "victim = self.running.pop()          # newest admitted",
     "victim = self.running.pop(0)", SCHED_PINS),
    ("sched_admit_after_preemption", SCHED, "if preempted == 0:", "if True:", SCHED_PINS),
    ("sched_preempted_to_queue_back", SCHED, "self.queue.insert(0, victim)",
     "self.queue.append(victim)", SCHED_PINS),
    ("sched_slot_offset", SCHED, "slots.append(r.table[pos // self.bs] * self.bs + pos % self.bs)",
     "slots.append(r.table[pos // self.bs] * self.bs + (pos + 1) % self.bs)", SCHED_PINS),
    ("sched_no_sampled_token", SCHED, "r.generated += 1", "r.generated += 0 if n > 1 else 1",
     SCHED_PINS),
]


def _copy_oracle(dst: str) -> str:
    pkg = os.path.join(dst, "oracle")
    os.makedirs(pkg)
    for name in (C, PY, SCHED):
        shutil.copy(os.path.join(ORACLE_DIR, name), os.path.join(pkg, name))
    return pkg


def _run_pins(pkg: str, pins) -> subprocess.CompletedProcess:
    env = dict(os.environ, PHOTON_ORACLE_UNDER_TEST=pkg)
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
           "-m", "not gpu"] + list(pins)
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def _plant(base: str, mutant) -> subprocess.CompletedProcess:
    name, fname, old, new, pins = mutant
    pkg = _copy_oracle(os.path.join(base, name))
    path = os.path.join(pkg, fname)
    src = open(path).read()
    assert src.count(old) == 1, f"{name}: the text to replace must occur once in {fname}"
    open(path, "w").write(src.replace(old, new))
    return _run_pins(pkg, pins)


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    base = str(tmp_path_factory.mktemp("oracle_mutants"))
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        control = ex.submit(lambda: _run_pins(_copy_oracle(os.path.join(base, "control")),
                                              PINS + ["tests/test_scheduler_cpu.py"]))
        futs = {m[0]: ex.submit(_plant, base, m) for m in MUTANTS}
        return control.result(), {k: f.result() for k, f in futs.items()}


def test_unmutated_copy_passes_every_pin(results):
    control, _ = results
    assert control.returncode == 0, control.stdout[-3000:] + control.stderr[-3000:]


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(results, name):
    control, runs = results
    assert control.returncode == 0
    r = runs[name]
    # pytest exits 1 when a test failed; anything else (2: an error while
    # collecting, 5: nothing collected) would mean the pins never ran
    assert r.returncode == 1, f"{name} survived the pins (exit {r.returncode}):\n" + \
        r.stdout[-2000:] + r.stderr[-2000:]
