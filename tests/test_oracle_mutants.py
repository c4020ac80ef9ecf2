"""The oracle's pins, run against deliberately broken copies of the oracle.

Each mutant below is one plausible slip in the oracle: an off-by-one, a
dropped term, a wrong sign, a transposed index, a misread layout.  It is
planted on the CPU, in a copy of the oracle's sources inside a temporary
directory.  The committed pins (tests/test_oracle_pins.py, unchanged) are then
run against that copy in a child process, and the mutant counts as killed when
a pin fails.  A mutant that survives means a pin is missing.  The repository's
own oracle is never modified.

The unmutated copy must pass first ("control"): otherwise a broken sandbox
would make every mutant look killed.
"""

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C = "oracle/dcp_oracle.c"
PY = "oracle/__init__.py"

# (name, file, text in the oracle, planted replacement).  The text must occur
# exactly once, so that an edit of the oracle cannot silently disarm a mutant.
MUTANTS = [
    # ownership and local layout
    ("rank_ignores_interleave", C,
     "return (t / I) % N; }", "return t % N; }"),
    ("rank_divides_by_virtual_block", C,
     "return (t / I) % N; }", "return (t / (I * N)) % N; }"),
    ("local_position_off_by_one", C,
     "lpos[t] = count[r]++;", "lpos[t] = ++count[r];"),
    ("local_length_counts_one_token_too_many", C,
     "for (int64_t t = 0; t < L; ++t) n += (orc_rank_of(t, N, I) == r);",
     "for (int64_t t = 0; t <= L; ++t) n += (orc_rank_of(t, N, I) == r);"),
    # block counts and slots
    ("virtual_block_ignores_ranks", C,
     "virt_blocks[b] = (int32_t)ceil_div(L, bs * N);", "virt_blocks[b] = (int32_t)ceil_div(L, bs);"),
    ("rank_blocks_rounded_down", C,
     "rank_blocks[r * B + b] = (int32_t)ceil_div(n, bs);", "rank_blocks[r * B + b] = (int32_t)(n / bs);"),
    ("slot_block_from_global_position", C,
     "int64_t blk = lp / bs;", "int64_t blk = p / bs;"),
    ("slot_offset_from_global_position", C,
     "slots[r_own * T + i] = (int64_t)id * bs + lp % bs;", "slots[r_own * T + i] = (int64_t)id * bs + p % bs;"),
    ("block_table_rank_and_request_transposed", C,
     "block_tables[(r_own * B + b) * max_blocks + blk]", "block_tables[(b * N + r_own) * max_blocks + blk]"),
    ("missing_block_id_not_reported", C,
     "if (id < 0) { status = -1; continue; }", "if (id < 0) { continue; }"),
    # PD block-transfer listing
    ("transfer_pool_bound_off_by_one", C,
     "if (id < 0 || id >= num_blocks) { status = -1; id = -1; }",
     "if (id < 0 || id > num_blocks) { status = -1; id = -1; }"),
    ("transfer_counts_tokens_as_slots", C,
     "totals[0] += bs;", "totals[0] += n;"),
    ("transfer_table_rank_and_request_transposed", C,
     "int32_t id = block_tables[(r * B + b) * max_blocks + k];",
     "int32_t id = block_tables[(b * N + r) * max_blocks + k];"),
    ("transfer_fill_as_full_block", C,
     "of[c] = (int32_t)n;", "of[c] = (int32_t)bs;"),
    ("transfer_lists_empty_blocks", C,
     "if (n == 0) continue;", ";"),
    ("transfer_tokens_counted_as_slots", C,
     "totals[1] += n;", "totals[1] += bs;"),
    # PCP head-tail partition
    ("pcp_padded_length_left_unpadded", C,
     "padded_len[b] = (int32_t)aligned;", "padded_len[b] = (int32_t)n;"),
    ("pcp_tail_chunk_not_mirrored", C,
     "const int64_t chunks[2] = {k, 2 * K - 1 - k};", "const int64_t chunks[2] = {k, K + k};"),
    ("pcp_aligns_to_K_not_2K", C,
     "const int64_t aligned = (n + 2 * K - 1) / (2 * K) * (2 * K);",
     "const int64_t aligned = (n + K - 1) / K * K;"),
    ("pcp_padding_not_marked", C,
     "row[out++] = rel < n ? (int32_t)(ctx_lens[b] + rel) : -1;", "row[out++] = (int32_t)(ctx_lens[b] + rel);"),
    ("pcp_capacity_off_by_one", C,
     "if (aligned > max_q) {", "if (aligned >= max_q) {"),
    ("pcp_positions_without_the_context", C,
     "row[out++] = rel < n ? (int32_t)(ctx_lens[b] + rel) : -1;", "row[out++] = rel < n ? (int32_t)(rel) : -1;"),
    ("pcp_tail_before_head", C,
     "const int64_t chunks[2] = {k, 2 * K - 1 - k};", "const int64_t chunks[2] = {2 * K - 1 - k, k};"),
    # storage decoding
    ("fp8_exponent_bias_8", C,
     "mag = ldexp(1.0 + (double)m / 8.0, e - 7);", "mag = ldexp(1.0 + (double)m / 8.0, e - 8);"),
    ("fp8_subnormal_scale", C,
     "mag = ldexp((double)m / 8.0, -6);", "mag = ldexp((double)m / 8.0, -7);"),
    ("fp8_per_tensor_scale_dropped", C,
     "return orc_fp8_e4m3_value(((const uint8_t*)base)[idx]) * scale;",
     "return orc_fp8_e4m3_value(((const uint8_t*)base)[idx]);"),
    ("fp8_nan_code_dropped", C,
     "if (e == 0xF && m == 0x7) return NAN;", ";"),
    # attention
    ("causal_bound_off_by_one", C,
     "int64_t g = L - Tq + t + 1;", "int64_t g = L - Tq + t;"),
    ("no_causal_mask_among_new_tokens", C,
     "int64_t g = L - Tq + t + 1;", "int64_t g = L;"),
    ("gqa_heads_interleaved_not_grouped", C,
     "int64_t kvh = h / group;", "int64_t kvh = h % Hkv;"),
    ("keys_without_rope_columns", C,
     "for (int64_t d = 0; d < Dk; ++d) dot += qv[d] * orc_load(k, row * Dk + d, kv_dtype, kv_scale);",
     "for (int64_t d = 0; d < Dv; ++d) dot += qv[d] * orc_load(k, row * Dk + d, kv_dtype, kv_scale);"),
    ("every_head_reads_the_first_heads_query", C,
     "qv[d] = orc_load(q, id * Dk + d, q_dtype, 1.0);", "qv[d] = orc_load(q, (id - h) * Dk + d, q_dtype, 1.0);"),
    ("softmax_scale_dropped", C,
     "s[cnt] = softmax_scale * dot;", "s[cnt] = dot;"),
    ("lse_drops_max_shift", C,
     "double L_row = m + log(sum);", "double L_row = log(sum);"),
    ("weights_not_normalised", C,
     "double w = exp(s[c] - L_row);", "double w = exp(s[c] - m);"),
    ("mla_values_are_last_columns", C,
     "o[d] += w * orc_load(k, idx[c] * Dk + d, kv_dtype, kv_scale);",
     "o[d] += w * orc_load(k, idx[c] * Dk + (Dk - Dv) + d, kv_dtype, kv_scale);"),
    ("rank_filter_inverted", C,
     "if (rank >= 0 && orc_rank_of(j, N, I) != rank) continue;",
     "if (rank >= 0 && orc_rank_of(j, N, I) == rank) continue;"),
    ("query_row_of_wrong_token", C,
     "int64_t t = (id / Hq) % Tq;", "int64_t t = (id / Hq) % Tq; t = Tq - 1 - t;"),
    ("kv_rows_ignore_request_offset", C,
     "int64_t row = (req_start[b] + j) * Hkv + kvh;", "int64_t row = j * Hkv + kvh;"),
    ("lse_in_base_2", C,
     "double L_row = m + log(sum);", "double L_row = m + log2(sum);"),
    # merge
    ("merge_max_starts_at_zero", C,
     "        double l = -INFINITY;\n        for (int64_t i = 0; i < N; ++i)",
     "        double l = 0.0;\n        for (int64_t i = 0; i < N; ++i)"),
    ("merge_all_empty_rows_not_special", C,
     "        if (l == -INFINITY) {\n            lse[n] = -INFINITY;\n            continue;\n        }", ""),
    ("merge_weight_sign_flipped", C,
     "double a = exp(lse_parts[i * rows + n] - l);", "double a = exp(l - lse_parts[i * rows + n]);"),
    ("merge_partials_indexed_rows_first", C,
     "o[d] += a * o_parts[(i * rows + n) * Dv + d];", "o[d] += a * o_parts[(n * N + i) * Dv + d];"),
    ("merge_lse_drops_log_sum", C,
     "lse[n] = l + log(asum);", "lse[n] = l;"),
    ("merge_output_not_normalised", C,
     "for (int64_t d = 0; d < Dv; ++d) o[d] /= asum;", ";"),
    ("attention_wrapper_swaps_N_and_I", PY,
     'float(wl.kv_scale), float(c["softmax_scale"]), int(c["N"]), int(c["I"]),',
     'float(wl.kv_scale), float(c["softmax_scale"]), int(c["I"]), int(c["N"]),'),
    # sparse (top-k) localisation and attention
    ("sparse_rows_token_major", PY,
     "            i = b * Tq + t\n            C = cand[i][cand[i] >= 0]",
     "            i = t * B + b\n            C = cand[i][cand[i] >= 0]"),
    ("sparse_localize_keeps_global_position", PY,
     "local[r, i, counts[r, i]] = lp[t]", "local[r, i, counts[r, i]] = t"),
    ("sparse_count_not_advanced", PY,
     "            counts[r, i] += 1", "            counts[r, i] = 1"),
    ("sparse_rank_filter_inverted", PY,
     "C = C[layouts[L][0][C] == rank]", "C = C[layouts[L][0][C] != rank]"),
    ("sparse_query_of_the_first_token", PY,
     'q = decode(wl.q[b, t], c["q_dtype"])', 'q = decode(wl.q[b, 0], c["q_dtype"])'),
    ("sparse_rows_without_request_offset", PY,
     "rows_kv = wl.req_start[b] + C", "rows_kv = C"),
    ("sparse_keys_without_rope_columns", PY,
     "s = scale * (kk[:, g, :] @ q[h])", "s = scale * (kk[:, g, :Dv] @ q[h, :Dv])"),
    ("sparse_gqa_heads_interleaved", PY,
     "g = h // G", "g = h % Hkv"),
    ("sparse_lse_drops_max_shift", PY,
     "lse[r] = m + np.log(l)", "lse[r] = np.log(l)"),
    ("sparse_output_not_normalised", PY,
     "out[r] = (w @ vv[:, g, :]) / l", "out[r] = w @ vv[:, g, :]"),
]


def _sandbox(tmp_path):
    """A copy of what the pins need: the oracle's sources, the seeded
    generator, the pins, their conftest and their golden files."""
    root = tmp_path / "repo"
    for d in ("oracle", "dcp_workloads"):
        os.makedirs(root / d)
        for name in os.listdir(os.path.join(ROOT, d)):
            if name.endswith((".py", ".c")):
                shutil.copy(os.path.join(ROOT, d, name), root / d / name)
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), root / "tests" / "golden")
    for name in ("conftest.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", name), root / "tests" / name)
    return root


def _run_pins(root):
    cmd = [sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q",
           "-p", "no:cacheprovider", "-m", "not gpu"]
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    return subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=600)


def _plant(tmp_root, name, path, text, planted):
    root = _sandbox(tmp_root)
    if name is not None:
        src = (root / path).read_text()
        if src.count(text) != 1:
            return None
        (root / path).write_text(src.replace(text, planted))
    return _run_pins(root)


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """Every mutant's pin run, the control's included, run side by side (each
    child process is independent; they share no files)."""
    cases = [("control", None, None, None)] + MUTANTS
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as pool:
        futs = {c[0]: pool.submit(_plant, tmp_path_factory.mktemp(c[0]), None if c[0] == "control" else c[0],
                                  c[1], c[2], c[3]) for c in cases}
        return {k: f.result() for k, f in futs.items()}


def test_control_copy_passes_every_pin(outcomes):
    r = outcomes["control"]
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_kill_mutant(outcomes, name):
    r = outcomes[name]
    assert r is not None, f"mutant {name}: its text no longer occurs exactly once in the oracle"
    out = r.stdout[-3000:] + r.stderr[-2000:]
    assert r.returncode != 0, f"mutant {name} survived every pin"
    # killed by a failing pin, not by a crash or a collection error
    assert r.returncode == 1 and " failed" in r.stdout, f"mutant {name} broke the run:\n{out}"
