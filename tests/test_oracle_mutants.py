"""Mutation check of the oracle's pins.

Each mutant is a copy of the oracle's C source with one plausible mistake
planted by an exact text substitution: a dropped term or factor, a wrong
sign, exponent bias or index, a transposed operand, a reversed tie-break.
The copy is compiled on the CPU in a temporary folder and the pin suite
(tests/test_oracle_pins.py) runs against it in a child process, through the
``MOE_ORACLE_MUTANT_SRC`` hook of the ``orc`` fixture.  Every mutant must make
at least one pin fail; an unmutated copy taken through the same route must
pass them all.  The oracle's own source is only read, never modified.
"""
import os
import re
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE_SRC = os.path.join(ROOT, "oracle", "moe_oracle.c")

# (name, text in the oracle source, replacement)
MUTANTS = [
    # number formats
    ("e2m1_exponent_bias", "ldexp(1.0 + 0.5 * m, e - 1)", "ldexp(1.0 + 0.5 * m, e)"),
    ("e2m1_subnormal_step", "(e == 0) ? 0.5 * m", "(e == 0) ? 1.0 * m"),
    ("e4m3_exponent_bias", "ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)"),
    ("e4m3_subnormal_scale", "ldexp(m / 8.0, -6)", "ldexp(m / 8.0, -7)"),
    ("e4m3_nan_code_decoded", "if (e == 15 && m == 7)", "if (0)"),
    ("bf16_round_truncates", "nearbyint(ldexp(a, -qexp))", "floor(ldexp(a, -qexp))"),
    ("bf16_round_extra_bit", "int qexp = e - 8;", "int qexp = e - 9;"),
    ("bf16_subnormal_quantum", "if (qexp < -133)              /* quantum of the bfloat16 subnormals */\n        qexp = -133;",
     "if (qexp < -132)              /* quantum of the bfloat16 subnormals */\n        qexp = -132;"),
    ("bf16_overflow_threshold", "if (q > 0x1.FEp127)", "if (q > 0x1.FCp127)"),
    ("bf16_nan_to_infinity", "return 0x7FC0;", "return 0x7F80;"),
    ("e2m1_sign_dropped", "    return sign ? -mag : mag;\n}\n\n/* FP8", "    return mag;\n}\n\n/* FP8"),
    # NVFP4 matrix layout
    ("nibble_order_swapped", "(k & 1) ? (byte >> 4) : (byte & 15)",
     "(k & 1) ? (byte & 15) : (byte >> 4)"),
    ("scale_block_of_32", "(size_t)(k / 16)]", "(size_t)(k / 32)]"),
    ("scale2_dropped", "return qs * m->scale2;", "return qs;"),
    # FP8 and BF16 expert matrices
    ("fp8_scale2_dropped", "float q = (float)orc_e4m3(m->packed[i]);\n        return q * m->scale2;",
     "float q = (float)orc_e4m3(m->packed[i]);\n        return q;"),
    ("fp8_row_stride_halved", "const size_t i = (size_t)n * (size_t)K + (size_t)k;",
     "const size_t i = (size_t)n * (size_t)(K / 2) + (size_t)k;"),
    ("bf16_bytes_swapped", "(uint16_t)(m->packed[2 * i] | ((unsigned)m->packed[2 * i + 1] << 8))",
     "(uint16_t)(m->packed[2 * i + 1] | ((unsigned)m->packed[2 * i] << 8))"),
    ("bf16_read_as_fp8", "    if (m->fmt == ORC_FMT_FP8) {", "    if (m->fmt != ORC_FMT_NVFP4) {"),
    ("scale_row_stride_halved", "m->scales[(size_t)n * (size_t)(K / 16)",
     "m->scales[(size_t)n * (size_t)(K / 32)"),
    ("packed_row_stride_halved", "m->packed[(size_t)n * (size_t)(K / 2)",
     "m->packed[(size_t)n * (size_t)(K / 4)"),
    # router
    ("router_transposed", "w->router_bf16[(size_t)e * H + h]",
     "w->router_bf16[(size_t)h * E + e]"),
    ("router_reads_row0", "orc_bf16(x[(size_t)r * H + h])", "orc_bf16(x[h])"),
    ("logits_transposed", "logits[(size_t)r * E + e] = acc;", "logits[(size_t)e * rows + r] = acc;"),
    ("router_dot_drops_last_input",
     "            for (int h = 0; h < H; ++h)\n                acc += xr[h] * wr[h];",
     "            for (int h = 0; h < H - 1; ++h)\n                acc += xr[h] * wr[h];"),
    ("nvfp4_router_row0", "mat_row(&w->router_fp4, H, e, wr);",
     "mat_row(&w->router_fp4, H, 0, wr);"),
    # top-k and routing weights
    ("topk_ties_to_higher_id", "key[e] > key[best]", "key[e] >= key[best]"),
    ("topk_repeats_an_expert", "            if (taken[e])\n                continue;\n", ""),
    ("softmax_key_in_fp64", "key[e] = (double)(float)logit[e];", "key[e] = logit[e];"),
    ("sigmoid_key_in_fp64", "key[e] = (double)(float)(score[e] + (double)w->bias[e]);",
     "key[e] = score[e] + (double)w->bias[e];"),
    ("softmax_selects_smallest", "key[e] = (double)(float)logit[e];",
     "key[e] = -(double)(float)logit[e];"),
    ("softmax_unnormalised", "score[e] = exp(logit[e] - mx) / z;",
     "score[e] = exp(logit[e] - mx);"),
    ("softmax_denominator_unshifted", "            z += exp(logit[e] - mx);",
     "            z += exp(logit[e]);"),
    ("weight_of_slot_not_expert", "        double v = score[ids[j]];", "        double v = score[j];"),
    ("norm_sum_drops_last_slot", "    for (int j = 0; j < k; ++j)\n        sum += score[ids[j]];",
     "    for (int j = 0; j + 1 < k; ++j)\n        sum += score[ids[j]];"),
    ("bias_of_mirrored_expert", "(double)(float)(score[e] + (double)w->bias[e]);",
     "(double)(float)(score[e] + (double)w->bias[E - 1 - e]);"),
    ("sigmoid_sign", "return 1.0 / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(z));"),
    ("sigmoid_bias_in_weights", "score[e] = sigmoid64(logit[e]);",
     "score[e] = sigmoid64(logit[e]) + (double)w->bias[e];"),
    ("sigmoid_bias_not_in_key",
     "key[e] = (double)(float)(score[e] + (double)w->bias[e]);",
     "key[e] = (double)(float)score[e];"),
    ("norm_over_all_experts", "for (int j = 0; j < k; ++j)\n        sum += score[ids[j]];",
     "for (int j = 0; j < E; ++j)\n        sum += score[j];"),
    ("norm_flag_ignored", "if (c->norm_topk_prob)\n            v /= sum;", "v /= sum;"),
    ("scaling_factor_dropped", "v *= c->routed_scaling_factor;", "v *= 1.0;"),
    # union
    ("union_keeps_duplicates", "if (uni[u] == ids[p]) {", "if (0 && uni[u] == ids[p]) {"),
    ("union_scan_skips_last_entry", "        for (int u = 0; u < U; ++u)\n            if (uni[u]",
     "        for (int u = 0; u + 1 < U; ++u)\n            if (uni[u]"),
    ("union_rowmask_slot_bit", "(1u << (p / k))", "(1u << (p % k))"),
    ("union_slot2u_last_entry", "slot2u[p] = (uint8_t)found;", "slot2u[p] = (uint8_t)(U - 1);"),
    ("union_rowmask_not_cleared", "            rowmask[U] = 0;\n", ""),
    # expert MLP
    ("silu_sign", "return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    ("swiglu_operands_swapped", "hbuf[i] = silu64(gs) * us;", "hbuf[i] = gs * silu64(us);"),
    ("up_reads_gate_matrix", "mat_row(u, H, i, row);", "mat_row(g, H, i, row);"),
    ("gate_dot_drops_last_input", "        for (int h = 0; h < H; ++h)\n            gs += row[h] * x[h];",
     "        for (int h = 0; h < H - 1; ++h)\n            gs += row[h] * x[h];"),
    ("down_dot_drops_last_input", "        for (int i = 0; i < I; ++i)\n            acc += row[i] * hbuf[i];",
     "        for (int i = 0; i < I - 1; ++i)\n            acc += row[i] * hbuf[i];"),
    ("down_row_wraps_at_inner_size", "mat_row(d, I, o, row);", "mat_row(d, I, o % I, row);"),
    # whole layer
    ("expert_ids_transposed", "int e = j->ids[(size_t)r * k + s];",
     "int e = j->ids[(size_t)s * j->rows + r];"),
    ("expert_reads_row0", "const double *xr = j->x + (size_t)r * H;", "const double *xr = j->x;"),
    ("shared_expert_truncated_to_moe_inter",
     "orc_expert_mlp(H, c->shared_inter, &j->w->sh_gate",
     "orc_expert_mlp(H, c->moe_inter < c->shared_inter ? c->moe_inter : c->shared_inter, "
     "&j->w->sh_gate"),
    ("shared_gate_negated", "gate = sigmoid64(dot);", "gate = sigmoid64(-dot);"),
    ("shared_gate_vector_elem0", "orc_bf16(w->sh_gate_vec[h])", "orc_bf16(w->sh_gate_vec[0])"),
    ("ungated_shared_halved", "gate = 1.0;", "gate = 0.5;"),
    ("weighted_sum_unweighted", "acc += wts[(size_t)r * k + j] * y[", "acc += y["),
    ("weighted_sum_drops_last_slot", "            for (int j = 0; j < k; ++j)\n                acc += wts",
     "            for (int j = 0; j + 1 < k; ++j)\n                acc += wts"),
    ("weighted_sum_slots_reversed", "y[((size_t)r * per_row + j) * H + o]",
     "y[((size_t)r * per_row + (k - 1 - j)) * H + o]"),
    ("shared_term_dropped", "acc += gate * y[", "acc += 0.0 * gate * y["),
    # the layer at caller-given experts
    ("given_ids_norm_flag_ignored", "v = c->norm_topk_prob ? v / tot : v;", "v = v / tot;"),
    ("given_ids_scaling_factor_dropped",
     "wsel[j] = c->scoring == 1 ? v * c->routed_scaling_factor : v;", "wsel[j] = v;"),
    ("given_ids_softmax_denominator_unshifted", "part += exp(logit[e] - top);",
     "part += exp(logit[e]);"),
    ("given_ids_weight_of_slot_not_expert", "double v = p[sel[j]];", "double v = p[j];"),
    ("given_ids_norm_sum_of_slots", "tot += p[sel[j]];", "tot += p[j];"),
    ("given_ids_sigmoid_sign", "p[e] = 1.0 / (1.0 + exp(-logit[e]));",
     "p[e] = 1.0 / (1.0 + exp(logit[e]));"),
    ("given_ids_rows_share_row0_weights", "orc_weights_for_ids(c, lg + (size_t)r * E, sel + (size_t)r * k,",
     "orc_weights_for_ids(c, lg + (size_t)r * E, sel,"),
    ("output_rounded_through_fp32", "out_bf16[(size_t)r * H + o] = orc_round_bf16(acc);",
     "out_bf16[(size_t)r * H + o] = orc_round_bf16((double)(float)acc);"),
]


def _mutate(src: str, old: str, new: str) -> str:
    assert src.count(old) == 1, "mutation site not unique: %r" % old
    return src.replace(old, new)


def _run_pins(folder: str, text: str):
    """Compile-check `text` as the oracle source in `folder`, run the pin
    suite against it; returns (returncode, first failing pin, output tail)."""
    os.makedirs(folder, exist_ok=True)
    src = os.path.join(folder, "moe_oracle.c")
    with open(src, "w") as f:
        f.write(text)
    syn = subprocess.run(["gcc", "-fsyntax-only", "-std=c11", "-D_DEFAULT_SOURCE", src],
                         capture_output=True, text=True)
    if syn.returncode != 0:
        return -1, None, syn.stderr[-2000:]
    # one thread per child: the children run side by side
    env = dict(os.environ, MOE_ORACLE_MUTANT_SRC=src, OMP_NUM_THREADS="1",
               OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    p = subprocess.run(
        [sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
         "-x", "-q", "-p", "no:cacheprovider", "-W", "ignore"],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    out = p.stdout + p.stderr
    m = re.search(r"FAILED \S+::(\S+)", out)
    return p.returncode, (m.group(1) if m else None), out[-2000:]


@pytest.fixture(scope="module")
def mutant_results(tmp_path_factory):
    base = tmp_path_factory.mktemp("oracle_mutants")
    with open(ORACLE_SRC) as f:
        src = f.read()
    jobs = {"unmutated": src}
    for name, old, new in MUTANTS:
        jobs[name] = _mutate(src, old, new)
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        futs = {name: ex.submit(_run_pins, str(base / name), text)
                for name, text in jobs.items()}
        return {name: fut.result() for name, fut in futs.items()}


def test_unmutated_copy_passes_the_pins(mutant_results):
    rc, failed, tail = mutant_results["unmutated"]
    assert rc == 0, tail


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_pins_reject_mutant(mutant_results, name):
    rc, failed, tail = mutant_results[name]
    assert rc != -1, "mutant does not compile:\n" + tail
    assert rc == 1 and failed is not None, "mutant %s survived the pins:\n%s" % (name, tail)
