"""Planted mistakes in the oracle must be caught by its pins.

Each case copies oracle/ring_oracle.c, plants one plausible mistake in the
copy (a wrong rounding rule, a rotation or chunk index off by one, a dropped
canonicalisation, a remainder given to the wrong chunks, a wrong scale), builds
it with the oracle's own flags, and runs the oracle's pin suites against it in
a child process (ORACLE_LIB points the oracle package at the copy).  Every
mutant must fail at least one pin: a mistake that all pins let through is one
the pins cannot tell from the method.  The unmutated copy must pass them all,
which also shows that the child really loads the copy.  Mistakes are planted in
the oracle, on the CPU; nothing here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = ["tests/test_oracle_pins.py", "tests/test_oracle_orders.py", "tests/test_oracle_compression.py"]

# (name, exact snippet of ring_oracle.c -- must occur once --, replacement)
MUTANTS = [
    # bf16 rounding
    ("bf16_ties_away_from_zero",
     "if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))", "if (dropped >= 0x8000u)"),
    ("bf16_truncates", "if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))", "if (0)"),
    ("bf16_nan_not_quieted", "return (uint16_t)((u >> 16) | 0x0040u);", "return (uint16_t)(u >> 16);"),
    ("hop_truncates_instead_of_rounding",
     "return narrow_bits(op_f32(widen_bits(local, dtype), widen_bits(incoming, dtype), op), dtype);",
     "return op_f32(widen_bits(local, dtype), widen_bits(incoming, dtype), op) >> (dtype == OR_BF16 ? 16 : 0);"),
    # the reduction operators
    ("nan_result_not_canonical", "    if (f32_bits_is_nan(r))\n        r = 0x7fffffffu;\n    return r;\n}",
     "    return r;\n}"),
    ("max_tie_gives_minus_zero", "r = a_bits & b_bits;", "r = a_bits | b_bits;"),
    ("min_tie_gives_plus_zero", "r = a_bits | b_bits; /* equal", "r = a_bits & b_bits; /* equal"),
    ("prod_adds", "r = f32_to_bits(a * b);", "r = f32_to_bits(a + b);"),
    ("avg_multiplies_by_reciprocal", "uint32_t r = f32_to_bits(x / (float)N);",
     "uint32_t r = f32_to_bits(x * (1.0f / (float)N));"),
    ("avg_divides_by_n_minus_1", "uint32_t r = f32_to_bits(x / (float)N);",
     "uint32_t r = f32_to_bits(x / (float)(N > 1 ? N - 1 : 1));"),
    # partition and schedule
    ("remainder_to_last_chunks", "len[c] = q + ((uint64_t)c < rem ? 1 : 0);",
     "len[c] = q + ((uint64_t)c >= (uint64_t)N - rem ? 1 : 0);"),
    ("schedule_ag_recv_off_by_one", "e[1] = mod((int64_t)i - s, N);", "e[1] = mod((int64_t)i - s - 1, N);"),
    ("schedule_source_is_right_neighbour", "e[2] = mod((int64_t)i - 1, N);", "e[2] = mod((int64_t)i + 1, N);"),
    ("rs_adds_into_wrong_chunk",
     "int c = mod((int64_t)i - 1 - s, N);\n            int src = mod((int64_t)i - 1, N);\n            const void *in",
     "int c = mod((int64_t)i - s, N);\n            int src = mod((int64_t)i - 1, N);\n            const void *in"),
    ("threaded_rs_adds_into_wrong_chunk",
     "int c = mod((int64_t)i - 1 - s, N);\n            const void *in = p->snap",
     "int c = mod((int64_t)i - s, N);\n            const void *in = p->snap"),
    ("ag_stores_wrong_chunk",
     "int c = mod((int64_t)i - s, N);\n            int src = mod((int64_t)i - 1, N);\n            memcpy((char *)buf[i]",
     "int c = mod((int64_t)i + 1 - s, N);\n            int src = mod((int64_t)i - 1, N);\n            memcpy((char *)buf[i]"),
    ("closed_form_rotation_off_by_one",
     "            uint32_t acc = contrib(load(in[c], dtype, e), N, dtype, op);\n            for (int k = 1; k < N; ++k)",
     "            uint32_t acc = contrib(load(in[(c + 1) % N], dtype, e), N, dtype, op);\n"
     "            for (int k = 2; k <= N; ++k)"),
    # the pre-multiplied AVG
    ("premul_skipped_in_closed_form", "return op == OR_AVGP ? premul(v, N, dtype) : v;", "return v;"),
    ("premul_divides_instead_of_multiplying",
     "uint32_t r = f32_to_bits(bits_to_f32(widen_bits(v, dtype)) * inv);",
     "uint32_t r = f32_to_bits(bits_to_f32(widen_bits(v, dtype)) / (float)N);"),
    # other schedules' orders
    ("hd_partner_not_xor", "void *partner = vb[v ^ (1 << k)];", "void *partner = vb[(v + (1 << k)) % pw];"),
    ("tree_levels_top_down",
     "    for (int k = 0; k < top; ++k)\n        for (int i = 0; i + (1 << k) < N; i += 1 << (k + 1))\n            for (uint64_t e",
     "    for (int k = top - 1; k >= 0; --k)\n        for (int i = 0; i + (1 << k) < N; i += 1 << (k + 1))\n            for (uint64_t e"),
    ("hier_representative_is_chunk_owner", "int rep = mod((int64_t)c - 1, L);", "int rep = c;"),
    # compression with error feedback
    ("int8_scale_over_128", "fcanon(amax / 127.0f)", "fcanon(amax / 128.0f)"),
    ("int8_ties_away_from_zero",
     "double r = frac > 0.5 ? f + 1.0 : frac < 0.5 ? f : (((int64_t)f & 1) ? f + 1.0 : f);",
     "double r = frac >= 0.5 ? f + 1.0 : f;"),
    ("int8_nan_ignored", "if (u[i] != u[i])\n                nan = 1;", "if (0)\n                nan = 1;"),
    ("residual_sign_flipped", "e[i] = fcanon(u[i] - v);\n            u[i] = v;\n        }\n    }",
     "e[i] = fcanon(v - u[i]);\n            u[i] = v;\n        }\n    }"),
    ("threshold_strict", "float v = u[i] >= threshold ? 1.0f : 0.0f;", "float v = u[i] > threshold ? 1.0f : 0.0f;"),
    ("topk_strict_threshold", "float v = (f32_to_bits(u[i]) & 0x7fffffffu) >= tau ? u[i] : 0.0f;",
     "float v = (f32_to_bits(u[i]) & 0x7fffffffu) > tau ? u[i] : 0.0f;"),
    ("topk_keeps_the_smallest", "return x < y ? 1 : (x > y ? -1 : 0);", "return x < y ? -1 : (x > y ? 1 : 0);"),
    ("topk_kth_off_by_one", "tau = mag[(k < K ? k : K) - 1];", "tau = mag[(k < K ? k : K - 1)];"),
    ("topk_residual_zeroed", "e[i] = fcanon(u[i] - v);\n        u[i] = v;\n    }\n    return OR_OK;",
     "e[i] = 0.0f;\n        u[i] = v;\n    }\n    return OR_OK;"),
    ("error_feedback_dropped",
     "u[i] = fcanon(bits_to_f32(widen_bits(load(grads[r], dtype, i), dtype)) + res[r][i]);",
     "u[i] = fcanon(bits_to_f32(widen_bits(load(grads[r], dtype, i), dtype)));"),
    # bucket fusion, AllToAllv, the halving-doubling pre-fold, hierarchical AVG, Reduce
    ("bucket_forward_order", "            for (int t = T - 1; t >= 0; --t) {", "            for (int t = 0; t < T; ++t) {"),
    ("alltoallv_recv_displacements_from_transposed_counts",
     "rd[(size_t)j * N + i] = o;\n            o += counts[(size_t)i * N + j];",
     "rd[(size_t)j * N + i] = o;\n            o += counts[(size_t)j * N + i];"),
    ("hd_prefold_adds_the_wrong_neighbour",
     "hop(load(buf[2 * v + 1], dtype, e), load(buf[2 * v], dtype, e), dtype, sop));",
     "hop(load(buf[2 * v + 1], dtype, e), load(buf[2 * v + 2], dtype, e), dtype, sop));"),
    ("hier_avg_divides_by_group_count", "scale_range(grp[g], soff[d], soff[d] + slen[d], N, dtype);",
     "scale_range(grp[g], soff[d], soff[d] + slen[d], G, dtype);"),
    ("reduce_takes_chunk_from_its_own_rank", "(char *)work[mod((int64_t)c - 1, N)] + off[c] * es, len[c] * es);",
     "(char *)work[c] + off[c] * es, len[c] * es);"),
    # the copy collectives and the compressors' edges
    ("gather_drops_the_last_rank",
     "    for (int r = 0; r < N; ++r)\n        memcpy((char *)out_root + off[r] * es, in[r], len[r] * es);",
     "    for (int r = 0; r < N - 1; ++r)\n        memcpy((char *)out_root + off[r] * es, in[r], len[r] * es);"),
    ("allgather_stores_from_the_right_neighbour",
     "int src = mod((int64_t)i - 1, N);\n            memcpy((char *)out[i] + off[c] * es, (char *)snap",
     "int src = mod((int64_t)i + 1, N);\n            memcpy((char *)out[i] + off[c] * es, (char *)snap"),
    ("int8_blocks_one_longer", "for (uint64_t b0 = 0; b0 < K; b0 += (uint64_t)block) {",
     "for (uint64_t b0 = 0; b0 < K; b0 += (uint64_t)block + 1) {"),
    ("topk_nan_ranked_lowest", "mag[i] = f32_to_bits(u[i]) & 0x7fffffffu;",
     "mag[i] = u[i] != u[i] ? 0u : f32_to_bits(u[i]) & 0x7fffffffu;"),
    ("chunk_offsets_ignore_the_remainder", "        off[c] = o;\n        o += len[c];",
     "        off[c] = (uint64_t)c * q;\n        o += len[c];"),
]


def _build_copy(tmp_path, name, snippet=None, repl=None):
    with open(oracle.SRC) as f:
        src = f.read()
    if snippet is not None:
        assert src.count(snippet) == 1, "snippet of %s must occur exactly once in ring_oracle.c" % name
        src = src.replace(snippet, repl)
    c = tmp_path / ("%s.c" % name)
    so = tmp_path / ("%s.so" % name)
    c.write_text(src)
    subprocess.run(["gcc"] + oracle.CFLAGS + ["-w", "-o", str(so), str(c)], check=True)
    return str(so)


def _run_pins(so):
    env = dict(os.environ, ORACLE_LIB=so)
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider"]
                          + PINS, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)


@pytest.fixture(scope="module")
def runs(tmp_path_factory):
    """Build every copy, then run the pin suites against all of them at once
    (independent child processes); each test below reads its own result."""
    from concurrent.futures import ThreadPoolExecutor

    tmp = tmp_path_factory.mktemp("mutants")
    libs = {"clean": _build_copy(tmp, "clean")}
    for name, snippet, repl in MUTANTS:
        libs[name] = _build_copy(tmp, name, snippet, repl)
    with ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
        futs = {name: ex.submit(_run_pins, so) for name, so in libs.items()}
        return {name: f.result() for name, f in futs.items()}


def test_unmutated_copy_passes_every_pin(runs):
    res = runs["clean"]
    assert res.returncode == 0, res.stdout[-3000:] + res.stderr[-2000:]


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(runs, name):
    res = runs[name]
    assert res.returncode == 1, "mutant %s passed every pin:\n%s" % (name, res.stdout[-2000:])
