"""Planted mistakes in the oracle must fail its pins.

Each case copies oracle/zero_oracle.cpp, plants one plausible mistake (a
dropped term, a wrong sign, bound, index or order, an off-by-one), compiles
the variant on the host, routes the oracle module through it and runs the
pins of tests/test_oracle_pins.py until one fails. A variant that passes every
pin would mean the pins cannot tell that mistake from the method. The oracle's
own source is never changed. CPU only.

Every edit keeps all memory accesses in bounds, and none is equivalent to the
original (an edit that cannot change any output is not a mistake).
"""
import inspect

import pytest

import oracle
import test_oracle_pins as pins

SRC = oracle.SRC_PATH

# (name, exact text in zero_oracle.cpp, replacement)
MUTANTS = [
    # casts
    ("encode_truncates", "std::nearbyint(std::ldexp(a, -quantum_exp))",
     "std::trunc(std::ldexp(a, -quantum_exp))"),
    ("encode_ties_away", "std::nearbyint(std::ldexp(a, -quantum_exp))",
     "std::round(std::ldexp(a, -quantum_exp))"),
    ("encode_no_subnormal_quantum", "const int quantum_exp = (e < emin ? emin : e) - f.man_bits;",
     "const int quantum_exp = e - f.man_bits;"),
    ("encode_overflow_bound", "if (r >= std::ldexp(1.0, emax + 1))", "if (r >= std::ldexp(1.0, emax + 2))"),
    ("decode_subnormal_exponent", "mag = std::ldexp((double)m, 1 - bias - f.man_bits);",
     "mag = std::ldexp((double)m, -bias - f.man_bits);"),
    ("load_formats_swapped", "return (float)decode_fmt(bits, dtype == ORC_F16 ? kF16 : kBF16);",
     "return (float)decode_fmt(bits, dtype == ORC_F16 ? kBF16 : kF16);"),
    ("encode_loses_negative_zero",
     "const uint32_t sign = std::signbit(x) ? (1u << (f.exp_bits + f.man_bits)) : 0u;",
     "const uint32_t sign = x < 0.0 ? (1u << (f.exp_bits + f.man_bits)) : 0u;"),
    ("decode_nan_as_inf", "mag = m ? NAN : INFINITY;", "mag = INFINITY;"),
    # a1 layout
    ("layout_last_bucket_unpadded",
     "  bucket_start[nb] = b0;\n  bucket_len[nb] = align_up(pos - b0, unit);\n  pos = b0",
     "  bucket_start[nb] = b0;\n  bucket_len[nb] = pos - b0;\n  pos = b0"),
    ("layout_align_32", "const int64_t kParamAlign = 64;", "const int64_t kParamAlign = 32;"),
    ("layout_pad_not_times_world", "const int64_t unit = (int64_t)world * kShardUnit;",
     "const int64_t unit = kShardUnit;"),
    ("layout_bucket_opens_early", "if (open_has_param && off + numel[p] - b0 > cap) {",
     "if (open_has_param && off + numel[p] - b0 >= cap) {"),
    # a2 reduce
    ("reduce_drops_last_rank", "for (int w = 1; w < world; ++w) s = s + load_f32(grads[w], i, grad_dtype);",
     "for (int w = 1; w < world - 1; ++w) s = s + load_f32(grads[w], i, grad_dtype);"),
    ("reduce_reverse_rank_order",
     "s = load_f32(grads[0], i, grad_dtype);\n"
     "      for (int w = 1; w < world; ++w) s = s + load_f32(grads[w], i, grad_dtype);",
     "s = load_f32(grads[world - 1], i, grad_dtype);\n"
     "      for (int w = world - 2; w >= 0; --w) s = s + load_f32(grads[w], i, grad_dtype);"),
    ("reduce_sums_in_fp64",
     "    float s = 0.0f;\n    if (real_mask == nullptr || real_mask[i]) {\n"
     "      s = load_f32(grads[0], i, grad_dtype);\n"
     "      for (int w = 1; w < world; ++w) s = s + load_f32(grads[w], i, grad_dtype);\n    }\n"
     "    store_rne(out, i - begin, comm_dtype, s);",
     "    double s = 0.0;\n    if (real_mask == nullptr || real_mask[i]) {\n"
     "      s = load_f32(grads[0], i, grad_dtype);\n"
     "      for (int w = 1; w < world; ++w) s = s + (double)load_f32(grads[w], i, grad_dtype);\n    }\n"
     "    store_rne(out, i - begin, comm_dtype, (float)s);"),
    ("reduce_reads_padding", "if (real_mask == nullptr || real_mask[i]) {", "if (true) {"),
    # a3 overflow
    ("overflow_ignores_nan", "if (!std::isfinite(r)) ovf = 1;", "if (std::isinf(r)) ovf = 1;"),
    ("sumsq_of_magnitudes", "acc += r * r;", "acc += std::fabs(r);"),
    # a4 norm and clip
    ("norm_without_sqrt", "info->grad_norm = inv * std::sqrt(norm_sq_raw);",
     "info->grad_norm = inv * norm_sq_raw;"),
    ("norm_ignores_divisor", "const double inv = 1.0 / (sc->scale * divisor);",
     "const double inv = 1.0 / sc->scale;"),
    ("clip_without_eps", "c = hp->max_grad_norm / (info->grad_norm + 1e-6);",
     "c = hp->max_grad_norm / info->grad_norm;"),
    ("clip_not_clamped", "if (c > 1.0) c = 1.0;", "if (c > 2.0) c = 2.0;"),
    ("gscale_ignores_clip", "info->gscale = inv * c;", "info->gscale = inv;"),
    # a5 loss-scale state machine
    ("no_backoff", "double s = sc->scale * sc->backoff_factor;", "double s = sc->scale;"),
    ("no_min_scale", "sc->scale = s < sc->min_scale ? sc->min_scale : s;", "sc->scale = s;"),
    ("counter_kept_on_overflow", "    sc->counter = 0;\n    return;\n  }", "    return;\n  }"),
    ("t_advances_on_skip", "    info->skipped = 1;\n    info->clip_coef = 0.0;",
     "    info->skipped = 1;\n    sc->t += 1;\n    info->clip_coef = 0.0;"),
    ("growth_one_step_early", "if (sc->dynamic && sc->counter == sc->growth_interval) {",
     "if (sc->dynamic && sc->counter == sc->growth_interval - 1) {"),
    ("counter_kept_after_growth",
     "    sc->scale = sc->scale * sc->growth_factor;\n    sc->counter = 0;",
     "    sc->scale = sc->scale * sc->growth_factor;"),
    ("growth_in_static_mode", "if (sc->dynamic && sc->counter == sc->growth_interval) {",
     "if (sc->counter == sc->growth_interval) {"),
    ("bc2_uses_beta1", "info->bc2 = 1.0 - std::pow(hp->beta2, (double)sc->t);",
     "info->bc2 = 1.0 - std::pow(hp->beta1, (double)sc->t);"),
    ("t_advanced_after_bias_correction",
     "  sc->t += 1;\n  info->bc1 = 1.0 - std::pow(hp->beta1, (double)sc->t);\n"
     "  info->bc2 = 1.0 - std::pow(hp->beta2, (double)sc->t);",
     "  info->bc1 = 1.0 - std::pow(hp->beta1, (double)(sc->t + (sc->t == 0)));\n"
     "  info->bc2 = 1.0 - std::pow(hp->beta2, (double)(sc->t + (sc->t == 0)));\n  sc->t += 1;"),
    # a6 AdamW
    ("no_bias_correction_1", "const double step_size = hp->lr / info->bc1;",
     "const double step_size = hp->lr;"),
    ("bias_correction_2_without_sqrt", "const double sqrt_bc2 = std::sqrt(info->bc2);",
     "const double sqrt_bc2 = info->bc2;"),
    ("eps_inside_sqrt", "const double denom = std::sqrt(vi) / sqrt_bc2 + hp->eps;",
     "const double denom = std::sqrt(vi / info->bc2 + hp->eps);"),
    ("no_weight_decay", "    p = p * (1.0 - hp->lr * hp->weight_decay);\n", ""),
    ("decay_scales_update_too", "    p = p - step_size * mi / denom;",
     "    p = p - (1.0 - hp->lr * hp->weight_decay) * step_size * mi / denom;"),
    ("momentum_sign", "mi = b1 * mi + (1.0 - b1) * g;", "mi = b1 * mi - (1.0 - b1) * g;"),
    ("betas_swapped", "mi = b1 * mi + (1.0 - b1) * g;", "mi = b2 * mi + (1.0 - b2) * g;"),
    ("second_moment_of_abs", "vi = b2 * vi + (1.0 - b2) * g * g;",
     "vi = b2 * vi + (1.0 - b2) * std::fabs(g);"),
    ("skipped_step_updates", "  if (info->skipped) return;\n  const double b1",
     "  const double b1"),
    # accumulation
    ("accumulate_ignores_first", "const float base = first ? 0.0f : main_grad[i];",
     "const float base = main_grad[i];"),
    ("accumulate_subtracts", "main_grad[i] = base + load_f32(micro, i, micro_dtype);",
     "main_grad[i] = base - load_f32(micro, i, micro_dtype);"),
    ("accumulate_writes_padding",
     "    if (real_mask != nullptr && !real_mask[i]) continue;\n    const float base = first",
     "    const float base = first"),
    # more scaler and update mistakes
    ("growth_applies_backoff", "    sc->scale = sc->scale * sc->growth_factor;",
     "    sc->scale = sc->scale * sc->backoff_factor;"),
    ("min_scale_comparison_flipped", "sc->scale = s < sc->min_scale ? sc->min_scale : s;",
     "sc->scale = s > sc->min_scale ? sc->min_scale : s;"),
    ("decay_without_lr", "    p = p * (1.0 - hp->lr * hp->weight_decay);",
     "    p = p * (1.0 - hp->weight_decay);"),
    ("divisor_ignored",
     "const double divisor = hp->grad_divisor > 0.0 ? hp->grad_divisor : (double)world;",
     "const double divisor = (double)world;"),
    ("encode_zero_shortcut_removed", "  if (n == 0.0) return sign;\n", ""),
    ("momentum_from_variance", "mi = b1 * mi + (1.0 - b1) * g;", "mi = b1 * vi + (1.0 - b1) * g;"),
    # composed ZeRO step
    ("norm_misses_last_rank", "    orc_overflow_sumsq(shard_grad[r].data(), comm_dtype, shard_total, "
     "shard_real.data(), &o, &s);\n    sumsq += s;",
     "    orc_overflow_sumsq(shard_grad[r].data(), comm_dtype, shard_total, "
     "shard_real.data(), &o, &s);\n    if (r + 1 < world) sumsq += s;"),
    ("stage1_reduces_without_mask", "      orc_reduce(grads, world, grad_dtype, 0, np, real.data(), "
     "comm_dtype, full.data());",
     "      orc_reduce(grads, world, grad_dtype, 0, np, nullptr, comm_dtype, full.data());"),
]


def _pin_calls():
    """Every pin of test_oracle_pins as a zero-argument callable, parametrized
    cases expanded (the exhaustive cast variant stays off)."""
    calls = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        grids = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if not grids:
            calls.append((name, lambda fn=fn: fn(oracle)))
            continue
        names, values = grids[0].args[0], grids[0].args[1]
        names = [n.strip() for n in names.split(",")] if isinstance(names, str) else list(names)
        for vals in values:
            vals = vals if isinstance(vals, (tuple, list)) else (vals,)
            kwargs = dict(zip(names, vals))
            calls.append((f"{name}{list(vals)}", lambda fn=fn, kw=kwargs: fn(oracle, **kw)))
    return calls


def test_every_mutant_edit_applies_once():
    src = open(SRC).read()
    for name, old, _ in MUTANTS:
        assert src.count(old) == 1, (name, src.count(old))
    assert len({m[0] for m in MUTANTS}) == len(MUTANTS)


def test_pins_pass_on_the_oracle_itself():
    for name, call in _pin_calls():
        call()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1
    path = tmp_path / f"{name}.cpp"
    path.write_text(src.replace(old, new))
    so = oracle.build_variant(str(path), str(tmp_path / f"lib{name}.so"))
    before = oracle.use_library(so)
    killed_by = None
    try:
        for pin, call in _pin_calls():
            try:
                call()
            except Exception:  # an assertion, or any error the variant causes
                killed_by = pin
                break
    finally:
        oracle.restore_library(before)
    assert killed_by is not None, f"no pin fails with the mistake '{name}' planted"
