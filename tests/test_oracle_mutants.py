"""Mutation check of the oracle's pins (CPU only).

Each case plants one plausible mistake in a copy of oracle/rcc_oracle.cpp (a
wrong operation order, a dropped term, a swapped coefficient, a wrong index),
builds it into a temporary library, and runs the pins against it: at least
one pin must fail.  This shows the pins are sharp enough to catch the mistake
rather than restating the code they check.  The oracle in the repository is
never modified.
"""
import ctypes as C
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "rcc_oracle.cpp")

# (name, text in the oracle, planted replacement, pins expected to catch it)
MUTANTS = [
    ("mean by reciprocal", "if (op == ORC_MEAN) acc = acc / (float)R;",
     "if (op == ORC_MEAN) acc = acc * (1.0f / (float)R);",
     [pins.test_mean_is_one_ieee_division]),
    ("fold in reverse rank order", "for (int r = 1; r < R; ++r) acc = acc + xs[r];\n    if (op == ORC_MEAN) acc = acc / (float)R;",
     "acc = xs[R - 1];\n    for (int r = R - 2; r >= 0; --r) acc = acc + xs[r];\n    if (op == ORC_MEAN) acc = acc / (float)R;",
     [pins.test_rank_order_fixes_rounding]),
    ("max keeps the later of equal values", "} else if (op == ORC_MAX ? (x > acc) : (x < acc)) {\n      acc = x;\n    }\n  }\n  return nan ? bits_f32",
     "} else if (op == ORC_MAX ? (x >= acc) : (x <= acc)) {\n      acc = x;\n    }\n  }\n  return nan ? bits_f32",
     [pins.test_max_min_special_values]),
    ("NaN not canonicalised", "return nan ? bits_f32(kCanonicalNaN) : acc;", "return acc;",
     [pins.test_max_min_special_values]),
    ("bf16 rounds half up", "uint32_t rounded = u + 0x7FFFu + lsb;", "uint32_t rounded = u + 0x8000u + 0u * lsb;",
     [pins.test_f32_to_bf16_matches_torch]),
    ("fp64->bf16 via fp32 (double rounding)", "  int e;\n  std::frexp(d, &e);",
     "  if (d == d) return orc_f32_to_bf16_rne((float)d);\n  int e;\n  std::frexp(d, &e);",
     [pins.test_f64_to_bf16_single_rounding]),
    ("reduce_scatter shard index reversed", "reduce_elements(R, dtype, op, send, (size_t)r * shard, shard, recv[r]);",
     "reduce_elements(R, dtype, op, send, (size_t)(R - 1 - r) * shard, shard, recv[r]);",
     [lambda orc: pins.test_collective_identities(orc, "f32", 4)]),
    ("all_gather writes at the receiver's slot", "static_cast<unsigned char*>(recv[r]) + (size_t)q * n_shard * es",
     "static_cast<unsigned char*>(recv[r]) + (size_t)((q + 1) % R) * n_shard * es",
     [lambda orc: pins.test_collective_identities(orc, "f32", 4)]),
    ("all_to_all takes the receiver's chunk from the wrong place",
     "static_cast<const unsigned char*>(send[q]) + (size_t)r * shard * es",
     "static_cast<const unsigned char*>(send[q]) + (size_t)q * shard * es",
     [lambda orc: pins.test_all_to_all_is_a_block_transpose(orc, 3, "f32")]),
    ("unscale dropped", "g[i] = mean * inv_scale;", "g[i] = mean;",
     [pins.test_mean_unscale_exact_on_integers]),
    ("non-finite not counted", "st->nonfinite += 1;\n      continue;", "continue;",
     [pins.test_stats_vs_fsum]),
    ("clip even below the threshold", "d->norm > max_grad_norm", "d->norm > 0.0",
     [pins.test_clip_decision]),
    ("no first-moment bias correction", "s->step_size = (float)(lr / bc1);", "s->step_size = (float)lr;",
     [pins.test_adamw_constant_gradient_closed_form]),
    ("no second-moment bias correction", "s->inv_bc2_sqrt = (float)(1.0 / std::sqrt(bc2));",
     "s->inv_bc2_sqrt = 1.0f;", [pins.test_adamw_constant_gradient_closed_form]),
    ("betas swapped in m", "float mi = s->beta1 * m[i] + s->one_minus_beta1 * gp;",
     "float mi = s->one_minus_beta1 * m[i] + s->beta1 * gp;",
     [pins.test_adamw_two_distinct_gradients_closed_form]),
    ("weight decay not applied", "float pi = p[i] * s->decay;", "float pi = p[i];",
     [pins.test_adamw_constant_gradient_closed_form]),
    ("eps inside the square root", "float denom = std::sqrt(vi) * s->inv_bc2_sqrt + s->eps;",
     "float denom = std::sqrt(vi + s->eps) * s->inv_bc2_sqrt;",
     [pins.test_adamw_constant_gradient_closed_form]),
    ("clip coefficient ignored", "float gp = g[i] * clip_coef;", "float gp = g[i];",
     [pins.test_adamw_first_step_with_clip]),
    ("scaler grows on overflow", "sc->scale *= sc->backoff_factor;", "sc->scale *= sc->growth_factor;",
     [pins.test_skip_on_nonfinite_and_scaler]),
    ("step counted when skipped", "  if (d->skip) {\n    orc_scaler_update(scaler, 1);\n    return;",
     "  if (d->skip) {\n    orc_scaler_update(scaler, 1);\n    *step += 1;\n    return;",
     [pins.test_skip_on_nonfinite_and_scaler]),
    ("report words swapped", "out[0] = (uint32_t)(u & 0xFFFFFFFFu);\n  out[1] = (uint32_t)(u >> 32);",
     "out[0] = (uint32_t)(u >> 32);\n  out[1] = (uint32_t)(u & 0xFFFFFFFFu);",
     [pins.test_report_pack_layout]),
    ("report count wraps", "(uint32_t)(st->nonfinite > 0xFFFFFFFFull ? 0xFFFFFFFFu : st->nonfinite)",
     "(uint32_t)st->nonfinite", [pins.test_report_pack_layout]),
    ("report drops the compensation", "  double s = orc_stats_value(st);\n  uint64_t u;",
     "  double s = st->sum;\n  uint64_t u;", [pins.test_report_pack_layout]),
    ("broadcast skips the last rank", "  for (int r = 0; r < R; ++r)\n    if (recv[r] != nullptr && recv[r] != root_send && bytes)",
     "  for (int r = 0; r < R - 1; ++r)\n    if (recv[r] != nullptr && recv[r] != root_send && bytes)",
     [lambda orc: pins.test_collective_identities(orc, "f32", 4)]),
    ("sum of squares without compensation", "    if (std::fabs(st->sum) >= std::fabs(x))\n      st->comp += (st->sum - t) + x;\n    else\n      st->comp += (x - t) + st->sum;",
     "", [pins.test_stats_vs_fsum]),
    ("scaler grows one step late", "if (sc->growth_tracker >= sc->growth_interval)",
     "if (sc->growth_tracker > sc->growth_interval)", [pins.test_scaler_growth_interval]),
    ("max/min miss a NaN after rank 0", "    float x = xs[r];\n    if (std::isnan(x)) {\n      nan = true;",
     "    float x = xs[r];\n    if (false) {\n      nan = true;", [pins.test_max_min_special_values]),
    ("bf16 widening drops the sign", "float orc_bf16_to_f32(uint16_t b) { return bits_f32((uint32_t)b << 16); }",
     "float orc_bf16_to_f32(uint16_t b) { return bits_f32((uint32_t)(b & 0x7FFFu) << 16); }",
     [pins.test_bf16_reduce_vs_torch_and_f64]),
]


def _build_mutant(tmp_path, src_text, i):
    cpp = tmp_path / f"mutant{i}.cpp"
    cpp.write_text(src_text)
    so = tmp_path / f"libmutant{i}.so"
    hdr_dir = os.path.dirname(SRC)
    subprocess.run(["g++", *oracle.build.CXXFLAGS, "-I", hdr_dir, str(cpp), "-o", str(so)],
                   check=True)
    lib = C.CDLL(str(so))
    oracle._declare(lib)
    return lib


@pytest.mark.parametrize("i", range(len(MUTANTS)), ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(orc, tmp_path, i):
    name, old, new, catchers = MUTANTS[i]
    text = open(SRC).read()
    assert text.count(old) == 1, "the oracle no longer contains the mutated line: " + name
    lib = _build_mutant(tmp_path, text.replace(old, new), i)
    saved = oracle._lib
    oracle._lib = lib
    try:
        caught = False
        for pin in catchers:
            try:
                pin(orc)
            except AssertionError:
                caught = True
        assert caught, "no pin caught the planted mistake: " + name
    finally:
        oracle._lib = saved
    # the real oracle still passes the same pins
    for pin in catchers:
        pin(orc)
