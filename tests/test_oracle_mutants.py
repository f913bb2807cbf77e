"""The oracle's pins catch plausible mistakes (CPU only).

Each case below plants one mistake in a copy of oracle/ep_oracle.c (a wrong
rounding rule, exponent bias or subnormal scale, another expert-to-rank map,
an inverted mask, a misplaced receive row, a reordered or double-rounded
sum, a wrong codec, a reversed gather), builds it with the oracle's own gcc
flags, and runs the oracle pin tests against it in a child process: at least
one pin must fail. The unchanged copy, built the same way, must pass. The
mistakes are planted in the oracle only, on the CPU.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "ep_oracle.c")
PINS = ["tests/test_oracle_formats.py", "tests/test_oracle_worked.py", "tests/test_oracle_invariants.py",
        "tests/test_oracle_bruteforce.py", "tests/test_oracle_eplb.py"]

COMBINE_ADD = """                    if (!oracle_routed_to(ids, top_k, num_experts, ep_size, d, mask_enabled,
                                          active_rank_mask))
                        continue;
                    acc = acc + oracle_bf16_to_f32(expert_output[d][r * hidden + h]);"""

# (name, text in ep_oracle.c, replacement)
MUTANTS = [
    ("bf16_ties_away", "if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u)))", "if (lo >= 0x8000u)"),
    ("bf16_truncates", "        hi += 1u;\n    return (uint16_t)hi;", "        hi += 0u;\n    return (uint16_t)hi;"),
    ("e4m3_bias", "for (int i = 7; i < e; ++i) mag = mag * 2.0f;", "for (int i = 8; i < e; ++i) mag = mag * 2.0f;"),
    ("e4m3_subnormal_scale", "for (int i = 0; i < 6; ++i) mag = mag / 2.0f;",
     "for (int i = 0; i < 7; ++i) mag = mag / 2.0f;"),
    ("f16_subnormal_scale", "for (int i = 0; i < 24; ++i) mag = mag / 2.0f;",
     "for (int i = 0; i < 23; ++i) mag = mag / 2.0f;"),
    ("f16_ties_away", "if (rem > half || (rem == half && (keep & 1u)))", "if (rem >= half)"),
    ("f16_overflow_early", "    if (e > 15)\n        return (uint16_t)(sign | 0x7C00u);",
     "    if (e > 14)\n        return (uint16_t)(sign | 0x7C00u);"),
    ("f16_subnormal_edge", "    if (e >= -14) {", "    if (e >= -15) {"),
    ("round_robin_owner", "if (e / experts_per_rank == d)\n            return 1;", "if (e % ep_size == d)\n            return 1;"),
    ("expert_zero_invalid", "        if (e < 0 || e >= num_experts)\n            continue;\n        if (e / experts_per_rank == d)",
     "        if (e <= 0 || e >= num_experts)\n            continue;\n        if (e / experts_per_rank == d)"),
    ("mask_inverted", "if (mask_enabled && !((active_rank_mask >> d) & 1u))", "if (mask_enabled && ((active_rank_mask >> d) & 1u))"),
    ("mask_ignored", "if (mask_enabled && !((active_rank_mask >> d) & 1u))", "if (0 && mask_enabled && !((active_rank_mask >> d) & 1u))"),
    ("invalid_id_zero", "                        id_row[k] = ORACLE_INVALID_EXPERT_ID;\n                    continue;",
     "                        id_row[k] = 0;\n                    continue;"),
    ("slot_order_transposed", "int32_t *id_row = recv_ids[d] + r * top_k;",
     "int32_t *id_row = recv_ids[d] + ((long)t * ep_size + s) * top_k;"),
    ("ids_only_owned", "id_row[k] = topk_ids[s][(long)t * top_k + k];",
     "id_row[k] = (topk_ids[s][(long)t * top_k + k] / (num_experts / ep_size) == d) ? "
     "topk_ids[s][(long)t * top_k + k] : ORACLE_INVALID_EXPERT_ID;"),
    ("scale_first_column_only", "recv_scale[d][r * scale_cols + j] = scale[s][(long)t * scale_cols + j];",
     "recv_scale[d][r * scale_cols + j] = scale[s][(long)t * scale_cols + 0];"),
    ("hidden_previous_row", "recv_hidden[d][r * row_bytes + b] = hidden[s][(long)t * row_bytes + b];",
     "recv_hidden[d][r * row_bytes + b] = hidden[s][(long)(t > 0 ? t - 1 : 0) * row_bytes + b];"),
    ("identity_scale_group_interleaved", "int group = h / (hidden / scale_cols);", "int group = h % scale_cols;"),
    ("scale_rows_need_two_columns", "if (scale_cols > 0 && scale && recv_scale && recv_scale[d])",
     "if (scale_cols > 1 && scale && recv_scale && recv_scale[d])"),
    ("e4m3_negative_nan_is_a_number", "if (e == 0xF && m == 0x7) {", "if (e == 0xF && m == 0x7 && sign == 0) {"),
    ("f16_nan_becomes_inf", "return (uint16_t)(sign | (man ? 0x7E00u : 0x7C00u));", "return (uint16_t)(sign | 0x7C00u);"),
    ("eplb_last_byte_dropped", "for (int b = 0; b < bytes; ++b)\n            global", "for (int b = 0; b + 1 < bytes; ++b)\n            global"),
    ("combine_skips_last_token", """    for (int s = 0; s < ep_size; ++s) {
        for (int t = 0; t < num_tokens[s]; ++t) {
            long r = (long)s * T + t;
            const int32_t *ids = topk_ids[s] + (long)t * top_k;
            for (int h = 0; h < hidden; ++h) {
                float acc = 0.0f;
                for (int d = 0; d < ep_size; ++d) {
""" + COMBINE_ADD, """    for (int s = 0; s < ep_size; ++s) {
        for (int t = 0; t + 1 < num_tokens[s]; ++t) {
            long r = (long)s * T + t;
            const int32_t *ids = topk_ids[s] + (long)t * top_k;
            for (int h = 0; h < hidden; ++h) {
                float acc = 0.0f;
                for (int d = 0; d < ep_size; ++d) {
""" + COMBINE_ADD),
    ("combine_skips_last_column", """            for (int h = 0; h < hidden; ++h) {
                float acc = 0.0f;
                for (int d = 0; d < ep_size; ++d) {
""" + COMBINE_ADD, """            for (int h = 0; h + 1 < hidden; ++h) {
                float acc = 0.0f;
                for (int d = 0; d < ep_size; ++d) {
""" + COMBINE_ADD),
    ("last_id_not_copied", """                for (int k = 0; k < top_k; ++k)
                    id_row[k] = topk_ids[s][(long)t * top_k + k];""", """                for (int k = 0; k + 1 < top_k; ++k)
                    id_row[k] = topk_ids[s][(long)t * top_k + k];"""),
    ("eplb_transposed", "global[(long)r * bytes + b] = local[r][b];", "global[(long)b * ep_size + r] = local[r][b];"),
    ("weights_reversed", "recv_weights[d][r * top_k + k] = topk_weights[s][(long)t * top_k + k];",
     "recv_weights[d][r * top_k + k] = topk_weights[s][(long)t * top_k + (top_k - 1 - k)];"),
    ("bf16_nan_sign_dropped", "return (uint16_t)(((u >> 16) & 0x8000u) | 0x7FC0u);", "return (uint16_t)0x7FC0u;"),
    ("mask_read_as_32_bits", "if (mask_enabled && !((active_rank_mask >> d) & 1u))",
     "if (mask_enabled && !(((uint32_t)active_rank_mask >> (d & 31)) & 1u))"),
    ("e4m3_sign_dropped", "    return sign ? -mag : mag;\n}\n\n/* IEEE 754 binary16", "    return mag;\n}\n\n/* IEEE 754 binary16"),
    ("f16_carry_lost", "uint32_t field = ((uint32_t)base_exp << 10) + (keep - 0x400u);",
     "uint32_t field = ((uint32_t)base_exp << 10) | (keep & 0x3FFu);"),
    ("identity_fp8_scale_ignored", """                    x = oracle_e4m3_to_f32(recv_hidden[d][r * hidden + h]) *
                        recv_scale[d][r * scale_cols + group];""", """                    x = oracle_e4m3_to_f32(recv_hidden[d][r * hidden + h]) *
                        (group >= 0 ? 1.0f : recv_scale[d][r * scale_cols + group]);"""),
    ("eplb_all_rows_from_rank0", "global[(long)r * bytes + b] = local[r][b];", "global[(long)r * bytes + b] = local[0][b];"),
    ("invalid_row_last_id_stale", """                    for (int k = 0; k < top_k; ++k)
                        id_row[k] = ORACLE_INVALID_EXPERT_ID;""", """                    for (int k = 0; k + 1 < top_k; ++k)
                        id_row[k] = ORACLE_INVALID_EXPERT_ID;"""),
    ("receive_row_without_source_offset", "recv_hidden[d][r * row_bytes + b] = hidden[s][(long)t * row_bytes + b];",
     "recv_hidden[d][(long)t * row_bytes + b] = hidden[s][(long)t * row_bytes + b];"),
    ("combine_reads_transposed_rows", "acc = acc + oracle_bf16_to_f32(expert_output[d][r * hidden + h]);",
     "acc = acc + oracle_bf16_to_f32(expert_output[d][((long)t * ep_size + s) * hidden + h]);"),
    ("f16_subnormal_shift_off_by_one", "shift = 13 + (-14 - e);  /* subnormal: grid of 2^-24 */",
     "shift = 14 + (-14 - e);  /* subnormal: grid of 2^-24 */"),
    ("identity_bf16_bytes_swapped", "x = oracle_bf16_to_f32((uint16_t)(p[0] | (p[1] << 8)));",
     "x = oracle_bf16_to_f32((uint16_t)((p[0] << 8) | p[1]));"),
    ("weights_not_copied", "recv_weights[d][r * top_k + k] = topk_weights[s][(long)t * top_k + k];",
     "recv_weights[d][r * top_k + k] = 0.0f;"),
    ("combine_descending", "                for (int d = 0; d < ep_size; ++d) {\n" + COMBINE_ADD,
     "                for (int d = ep_size - 1; d >= 0; --d) {\n" + COMBINE_ADD),
    ("combine_rounds_each_add", "acc = acc + oracle_bf16_to_f32(expert_output[d][r * hidden + h]);",
     "acc = oracle_bf16_to_f32(oracle_f32_to_bf16_rne(acc + oracle_bf16_to_f32(expert_output[d][r * hidden + h])));"),
    ("combine_all_ranks", COMBINE_ADD, COMBINE_ADD.replace("if (!oracle_routed_to", "if (0 && !oracle_routed_to")),
    ("combine_minus_zero_start", "                float acc = 0.0f;\n                for (int d = 0; d < ep_size; ++d) {\n" + COMBINE_ADD,
     "                float acc = -0.0f;\n                for (int d = 0; d < ep_size; ++d) {\n" + COMBINE_ADD),
    ("typed_f16_as_bf16", "x = oracle_f16_to_f32(((const uint16_t *)expert_output[d])[i]);",
     "x = oracle_bf16_to_f32(((const uint16_t *)expert_output[d])[i]);"),
    ("typed_f32_rounded", "((float *)out[s])[o] = acc;", "((float *)out[s])[o] = oracle_bf16_to_f32(oracle_f32_to_bf16_rne(acc));"),
    ("eplb_reversed", "global[(long)r * bytes + b] = local[r][b];", "global[(long)r * bytes + b] = local[ep_size - 1 - r][b];"),
    ("identity_last_weight", "w = w + (recv_weights ? recv_weights[d][r * top_k + k] : 1.0f);",
     "w = (recv_weights ? recv_weights[d][r * top_k + k] : 1.0f);"),
]


def _build(tmp_dir, name, text):
    c = os.path.join(tmp_dir, f"{name}.c")
    with open(c, "w") as f:
        f.write(text)
    so = os.path.join(tmp_dir, f"{name}.so")
    # the oracle's own flags (oracle/__init__.py)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
                           "-Wall", "-Wextra", "-o", so, c])
    return so


def _run_pins(so):
    env = dict(os.environ, EP_ORACLE_LIB=so)
    return subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", "-m", "not gpu",
                           *PINS], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)


@pytest.fixture(scope="module")
def pin_runs(tmp_path_factory):
    """Builds the unchanged copy and every mutant, and runs the pins against
    all of them at once (child processes in parallel): name -> result."""
    import concurrent.futures as cf
    tmp = str(tmp_path_factory.mktemp("oracle_mutants"))
    src = open(SRC).read()
    texts = {"control": src}
    for name, orig, mutated in MUTANTS:
        assert src.count(orig) == 1, f"{name}: the oracle no longer contains the text this mistake replaces"
        texts[name] = src.replace(orig, mutated)
    libs = {name: _build(tmp, name, text) for name, text in texts.items()}
    with cf.ThreadPoolExecutor(max_workers=max(2, min(16, os.cpu_count() or 2))) as ex:
        futures = {name: ex.submit(_run_pins, so) for name, so in libs.items()}
        return {name: f.result() for name, f in futures.items()}


def test_unchanged_copy_passes_the_pins(pin_runs):
    r = pin_runs["control"]
    assert r.returncode == 0, r.stdout[-3000:]


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(pin_runs, name):
    r = pin_runs[name]
    assert r.returncode != 0, f"{name}: every pin passed with the mistake planted"
    assert "failed" in r.stdout or r.returncode < 0, r.stdout[-2000:]
