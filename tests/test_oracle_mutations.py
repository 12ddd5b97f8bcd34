"""The oracle's pins against planted mistakes (CPU only).

Each case copies the oracle's C source, plants one plausible mistake in the copy (a wrong bit order,
a dropped offset or renormalisation, swapped or transposed matrices, a flipped tie rule, ...),
compiles the copy into a scratch library with the oracle's own flags, and runs
tests/test_oracle_pins.py against that library in a child process: the pins must fail.  The
unchanged copy, built the same way, must pass them.  Nothing here touches the real oracle library
or the GPU path.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "strata_oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, text in the oracle, planted replacement); each text occurs exactly once
MUTATIONS = [
    ("q2_bit_order_msb_first",
     "return (codes16[i >> 2] >> (2 * (i & 3))) & 3;",
     "return (codes16[i >> 2] >> (6 - 2 * (i & 3))) & 3;"),
    ("q2_code_byte_order",
     "return (codes16[i >> 2] >> (2 * (i & 3))) & 3;",
     "return (codes16[(i >> 2) ^ 1] >> (2 * (i & 3))) & 3;"),
    ("dequant_blocks_offset_dropped",
     "w[64 * b + i] = d * (double)(oracle_q2_code(blk + 2, i) - q2_offset);",
     "w[64 * b + i] = d * (double)(oracle_q2_code(blk + 2, i));"),
    ("expert_offset_sign",
     "return d * (double)(oracle_q2_code(blk + 2, (int)(flat % 64)) - q2_offset);",
     "return d * (double)(oracle_q2_code(blk + 2, (int)(flat % 64)) + q2_offset);"),
    ("expert_scale_bytes_swapped",
     "const double d = oracle_fp16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));\n  return d",
     "const double d = oracle_fp16_to_double((uint16_t)(blk[1] | (blk[0] << 8)));\n  return d"),
    ("fp16_exponent_bias",
     "v = ldexp((double)(man | 0x400), exp - 25);",
     "v = ldexp((double)(man | 0x400), exp - 24);"),
    ("bf16_low_half",
     "c.u = (uint32_t)b << 16;",
     "c.u = (uint32_t)b << 15;"),
    ("gate_up_swapped",
     "const uint8_t* gate = blob;\n  const uint8_t* up = blob + 18 * nb;",
     "const uint8_t* up = blob;\n  const uint8_t* gate = blob + 18 * nb;"),
    ("silu_on_up",
     "hbuf[r] = g / (1.0 + exp(-g)) * u;",
     "hbuf[r] = u / (1.0 + exp(-u)) * g;"),
    ("sigmoid_sign",
     "hbuf[r] = g / (1.0 + exp(-g)) * u;",
     "hbuf[r] = g / (1.0 + exp(g)) * u;"),
    ("down_transposed",
     "acc += q2_weight(down, FF, n, r, q2_offset) * hbuf[r];",
     "acc += q2_weight(down, H, r, n, q2_offset) * hbuf[r];"),
    ("router_bias_dropped",
     "if (bias) acc += (double)bias[e];",
     "(void)bias;"),
    ("top_k_ties_to_higher_id",
     "if (best < 0 || p[e] > p[best]) best = e;",
     "if (best < 0 || p[e] >= p[best]) best = e;"),
    ("top_k_not_renormalised",
     "for (int k = 0; k < K; ++k) w[k] = p[ids[k]] / denom;\n  if (p_out)",
     "for (int k = 0; k < K; ++k) w[k] = p[ids[k]];\n  if (p_out)"),
    ("group_unstable_order",
     "for (int p = 0; p < T * K; ++p) {\n    const int e = ids[p];",
     "for (int p = T * K - 1; p >= 0; --p) {\n    const int e = ids[p];"),
    ("rmsnorm_without_mean",
     "const double inv = 1.0 / sqrt(ss / (double)H + eps);",
     "const double inv = 1.0 / sqrt(ss + eps);"),
    ("router_on_raw_input",
     "oracle_router_logits(xn, H, E, j->w_router, j->bias, logits);\n  if (j->ids_in)",
     "oracle_router_logits(xin, H, E, j->w_router, j->bias, logits);\n  if (j->ids_in)"),
    ("route_tokens_rmsnorm_dropped",
     "if (j->residual) oracle_rmsnorm(xn, j->H, 1e-6, xn);",
     "(void)0;"),
    ("route_tokens_bias_dropped",
     "oracle_router_logits(xn, j->H, j->E, j->w_router, j->bias, logits);\n    oracle_top_k",
     "oracle_router_logits(xn, j->H, j->E, j->w_router, NULL, logits);\n    oracle_top_k"),
    ("shared_expert_dropped",
     "for (int h = 0; h < H; ++h) acc[h] += y[h];\n    }\n    if (!rc && j->residual)",
     "(void)0;\n    }\n    if (!rc && j->residual)"),
    ("shared_expert_on_raw_input",
     "oracle_expert(j->shared_blob, H, j->FF, j->q2_offset, xn, y);",
     "oracle_expert(j->shared_blob, H, j->FF, j->q2_offset, xin, y);"),
    ("shared_expert_weighted_by_first_router_weight",
     "for (int h = 0; h < H; ++h) acc[h] += y[h];\n    }\n    if (!rc && j->residual)",
     "for (int h = 0; h < H; ++h) acc[h] += w[0] * y[h];\n    }\n    if (!rc && j->residual)"),
    ("combine_unweighted",
     "for (int h = 0; h < H; ++h) acc[h] += w[k] * y[h];",
     "for (int h = 0; h < H; ++h) acc[h] += y[h];"),
    ("residual_dropped",
     "for (int h = 0; h < H; ++h) acc[h] = xin[h] + acc[h];",
     "for (int h = 0; h < H; ++h) acc[h] = acc[h];"),
    ("residual_added_to_the_normalised_input",
     "for (int h = 0; h < H; ++h) acc[h] = xin[h] + acc[h];",
     "for (int h = 0; h < H; ++h) acc[h] = xn[h] + acc[h];"),
    ("router_rows_transposed",
     "    const uint16_t* row = w_router + (int64_t)e * H;\n    for (int h = 0; h < H; ++h) acc += oracle_bf16_to_double(row[h]) * xn[h];",
     "    for (int h = 0; h < H; ++h) acc += oracle_bf16_to_double(w_router[(int64_t)h * E + e]) * xn[h];"),
    ("up_and_down_regions_swapped",
     "  const uint8_t* up = blob + 18 * nb;\n  const uint8_t* down = blob + 36 * nb;",
     "  const uint8_t* down = blob + 18 * nb;\n  const uint8_t* up = blob + 36 * nb;"),
    ("gate_transposed",
     "      g += q2_weight(gate, H, r, c, q2_offset) * x[c];",
     "      g += q2_weight(gate, FF, c, r, q2_offset) * x[c];"),
    ("swiglu_without_up",
     "hbuf[r] = g / (1.0 + exp(-g)) * u;",
     "hbuf[r] = g / (1.0 + exp(-g));"),
    ("experts_on_raw_input",
     "      oracle_expert(blob, H, j->FF, j->q2_offset, xn, y);",
     "      oracle_expert(blob, H, j->FF, j->q2_offset, xin, y);"),
    ("rmsnorm_epsilon_in_layer",
     "    oracle_rmsnorm(xin, H, 1e-6, xn);",
     "    oracle_rmsnorm(xin, H, 1e-5, xn);"),
    ("rmsnorm_epsilon_in_route",
     "if (j->residual) oracle_rmsnorm(xn, j->H, 1e-6, xn);",
     "if (j->residual) oracle_rmsnorm(xn, j->H, 1e-5, xn);"),
    ("forced_ids_not_renormalised",
     "  for (int k = 0; k < K; ++k) w[k] = p[ids[k]] / denom;\n  free(p);\n}",
     "  for (int k = 0; k < K; ++k) w[k] = p[ids[k]];\n  free(p);\n}"),
    ("forced_ids_all_take_the_first_weight",
     "  for (int k = 0; k < K; ++k) w[k] = p[ids[k]] / denom;\n  free(p);\n}",
     "  for (int k = 0; k < K; ++k) w[k] = p[ids[0]] / denom;\n  free(p);\n}"),
    ("parts_stored_slot_major",
     "memcpy(j->parts_out + ((int64_t)t * K + k) * H",
     "memcpy(j->parts_out + ((int64_t)k * j->T + t) * H"),
    ("active_list_descending",
     "  for (int e = 0; e < E; ++e)\n    if (count[e]) active[na++] = e;",
     "  for (int e = E - 1; e >= 0; --e)\n    if (count[e]) active[na++] = e;"),
]

# the child process: load the scratch library in place of the oracle's, then run the pins
RUNNER = ("import sys, oracle; oracle.LIB_PATH = sys.argv[1]; import pytest; "
          "sys.exit(pytest.main(['-x', '-q', '-p', 'no:cacheprovider', sys.argv[2]]))")


def build_copy(text, out_dir, name):
    c_path = os.path.join(out_dir, name + ".c")
    so_path = os.path.join(out_dir, "lib" + name + ".so")
    with open(c_path, "w") as f:
        f.write(text)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread",
           "-I", os.path.join(ROOT, "oracle"), "-o", so_path, c_path, "-lm"]
    subprocess.run(cmd, check=True)
    return so_path


def run_pins(so_path):
    env = dict(os.environ)
    env["PYTHONPATH"] = ROOT + os.pathsep + os.path.join(ROOT, "tests") + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", RUNNER, so_path, PINS], cwd=ROOT, env=env,
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True, timeout=600)
    return r.returncode, r.stdout


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


def test_unchanged_copy_passes_the_pins(source, tmp_path):
    rc, out = run_pins(build_copy(source, str(tmp_path), "unchanged"))
    assert rc == 0, out[-2000:]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(source, tmp_path, name, old, new):
    assert source.count(old) == 1, f"{name}: the text to replace is not unique in the oracle"
    rc, out = run_pins(build_copy(source.replace(old, new), str(tmp_path), name))
    assert rc == 1, f"{name}: the pins did not fail (exit {rc})\n{out[-2000:]}"
