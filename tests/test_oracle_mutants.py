"""Each plausible mistake planted in a copy of the oracle's source (a dropped
term, a wrong sign, index or order, a transposed operand) must fail at least
one pin. The mistakes are planted only in temporary CPU builds of the oracle;
the real oracle is untouched."""
import os
import subprocess

import pytest

import oracle
import pins

MUTANTS = [
    ("m sign", "m = m_prev_term + g_term;", "m = m_prev_term - g_term;"),
    ("beta2 in m", "float m_prev_term = s.b1 * m;", "float m_prev_term = s.b2 * m;"),
    ("beta1 in v", "float v_prev_term = s.b2 * v;", "float v_prev_term = s.b1 * v;"),
    ("v uses g not g^2", "float g_sq_term = g_scaled * g;", "float g_sq_term = g_scaled;"),
    ("1-beta1 in v", "s.omb2 = (float)(1.0 - beta2);", "s.omb2 = (float)(1.0 - beta1);"),
    ("bias corrections swapped", "float m_hat = m / s.bc1;", "float m_hat = m / s.bc2;"),
    ("bias correction one step late", "s.bc1 = (float)(1.0 - power_by_squaring(beta1, t));",
     "s.bc1 = (float)(1.0 - power_by_squaring(beta1, t + 1));"),
    ("eps inside sqrt", "float denom = std::sqrt(v_hat) + s.eps;",
     "float denom = std::sqrt(v_hat + s.eps);"),
    ("no weight decay", "float decayed = p * s.decay;", "float decayed = p;"),
    ("decay not scaled by lr", "s.decay = (float)(1.0 - lr * wd);", "s.decay = (float)(1.0 - wd);"),
    ("no learning rate", "float step = s.lr * update;", "float step = update;"),
    ("sum, not mean", "float g = acc * s.invN;", "float g = acc;"),
    ("descending reduce order",
     "for (int32_t j = 0; j < world; ++j) acc = acc + load_grad(grads[j], grad_dtype, i);",
     "for (int32_t j = world - 1; j >= 0; --j) acc = acc + load_grad(grads[j], grad_dtype, i);"),
    ("fp32 grads read as bf16", "return static_cast<const float*>(base)[i];",
     "return bf16_to_float(static_cast<const uint16_t*>(base)[i]);"),
    ("own slot at 0", "int64_t slot = (int64_t)rank * S;", "int64_t slot = 0;"),
    ("ties away from zero", "if (low > half || (low == half && (keep & 1u))) keep += 1u;",
     "if (low >= half) keep += 1u;"),
    ("NaN flushed", "return (sign | 0x7FC00000u) >> drop;", "return 0u;"),
    ("3-byte big-endian",
     "d[0] = (uint8_t)(q & 0xFFu);\n    d[1] = (uint8_t)((q >> 8) & 0xFFu);\n"
     "    d[2] = (uint8_t)((q >> 16) & 0xFFu);",
     "d[2] = (uint8_t)(q & 0xFFu);\n    d[1] = (uint8_t)((q >> 8) & 0xFFu);\n"
     "    d[0] = (uint8_t)((q >> 16) & 0xFFu);"),
    ("over-padding", "int64_t P_pad = (P + Q - 1) / Q * Q;", "int64_t P_pad = P / Q * Q + Q;"),
    ("ties ignored", "if (k < 0) {\n      owner[i] = i;", "if (true) {\n      owner[i] = i;"),
    ("offset after the tensor", "offsets[i] = P;\n      P += numels[i];",
     "P += numels[i];\n      offsets[i] = P;"),
    ("bucket closes one early", "if (cur_size > 0 && cur_size + n > bucket_elems) {",
     "if (cur_size > 0 && cur_size + n >= bucket_elems) {"),
    ("shard range short", "b = fhi - (int64_t)rank * S;", "b = fhi - (int64_t)rank * S - 1;"),
    ("ZeRO-2 keeps full grads", "case 2: return full_params + 2 * S + (4 + 4 + 4) * S;",
     "case 2: return full_params + 2 * P_pad + (4 + 4 + 4) * S;"),
    ("gather slot ignores element size",
     "static_cast<uint8_t*>(full_flat) + (size_t)j * S * elem_size, shards[j],",
     "static_cast<uint8_t*>(full_flat) + (size_t)j * S, shards[j],"),
    ("DDP sum, not mean", "mean[i] = acc * s.invN;", "mean[i] = acc;"),
    ("norm of the sum, not the mean", "float g = acc * invN;\n    sum = sum + (double)g * (double)g;",
     "float g = acc;\n    sum = sum + (double)g * (double)g;"),
    ("norm without square root", "double norm = std::sqrt(total);", "double norm = total;"),
    ("coefficient not clamped", "*coef = *nonfinite ? 1.0f : (float)(c < 1.0 ? c : 1.0);",
     "*coef = *nonfinite ? 1.0f : (float)c;"),
    ("non-finite never flagged", "*nonfinite = std::isfinite(norm) ? 0 : 1;", "*nonfinite = 0;"),
    ("skip ignored", "  if (skip) return 0;", "  if (false) return 0;"),
    ("coefficient ignored", "float g = (acc * s.invN) * coef;", "float g = acc * s.invN;"),
    ("accumulator overwritten every micro-step",
     "accum[i] = (first ? 0.0f : accum[i]) + mean;", "accum[i] = 0.0f + mean;"),
    ("first micro-step adds stale contents",
     "accum[i] = (first ? 0.0f : accum[i]) + mean;", "accum[i] = accum[i] + mean;"),
    ("accumulated gradient not divided by G", "float g = (accum[i] + mean) * invG;",
     "float g = accum[i] + mean;"),
    ("accumulator ignored by the step", "float g = (accum[i] + mean) * invG;",
     "float g = mean * invG;"),
    ("accumulated norm over the last micro-step only",
     "float g = (accum[i] + mean) * invG;\n    sum = sum + (double)g * (double)g;",
     "float g = mean * invG;\n    sum = sum + (double)g * (double)g;"),
    ("accumulated norm not divided by G",
     "float g = (accum[i] + mean) * invG;\n    sum = sum + (double)g * (double)g;",
     "float g = accum[i] + mean;\n    sum = sum + (double)g * (double)g;"),
    ("accumulated clip coefficient ignored", "float g = ((accum[i] + mean) * invG) * coef;",
     "float g = (accum[i] + mean) * invG;"),
    ("coefficient applied to the last micro-step only",
     "float g = ((accum[i] + mean) * invG) * coef;", "float g = (accum[i] + mean * coef) * invG;"),
    ("accumulated skip ignored",
     "  if (skip) return 0;\n  Scalars s = make_scalars(lr, beta1, beta2, eps, wd, t, world);\n"
     "  float invG",
     "  if (false) return 0;\n  Scalars s = make_scalars(lr, beta1, beta2, eps, wd, t, world);\n"
     "  float invG"),
    ("row chunks rounded down", "rows_per_rank[i] = (dim0[i] + world - 1) / world;",
     "rows_per_rank[i] = dim0[i] / world + (dim0[i] % world > 1 ? 1 : 0);"),
    ("segment offsets count rows, not elements",
     "local += rows_per_rank[i] * row_elems[i];", "local += rows_per_rank[i];"),
    ("local padding left uninitialised",
     "std::memset(local, 0, (size_t)S * elem_size);", "(void)0;"),
    ("3-byte range cast big-endian",
     "out[3 * i] = (uint8_t)(q & 0xFFu);\n    out[3 * i + 1] = (uint8_t)((q >> 8) & 0xFFu);\n"
     "    out[3 * i + 2] = (uint8_t)((q >> 16) & 0xFFu);",
     "out[3 * i + 2] = (uint8_t)(q & 0xFFu);\n    out[3 * i + 1] = (uint8_t)((q >> 8) & 0xFFu);\n"
     "    out[3 * i] = (uint8_t)((q >> 16) & 0xFFu);"),
    ("range cast one pattern ahead",
     "uint32_t q = round_keep_high(bits_float(first + (uint32_t)i), 8);",
     "uint32_t q = round_keep_high(bits_float(first + (uint32_t)i + 1u), 8);"),
    ("bf16 range cast one pattern ahead",
     "out[i] = (uint16_t)round_keep_high(bits_float(first + (uint32_t)i), 16);",
     "out[i] = (uint16_t)round_keep_high(bits_float(first + (uint32_t)i + 1u), 16);"),
    ("copy-out ignores the rank's row offset",
     "uint8_t* dst = static_cast<uint8_t*>(params[i]) + (size_t)r * rows_per_rank[i] * row_bytes;",
     "uint8_t* dst = static_cast<uint8_t*>(params[i]) + (size_t)r * row_bytes;"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new):
    src = open(oracle.SRC, encoding="utf-8").read()
    assert src.count(old) >= 1, f"mutation site not found: {old!r}"
    mutated = src.replace(old, new, 1)
    path = tmp_path / "oracle_mutant.cpp"
    path.write_text(mutated, encoding="utf-8")
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(oracle.build_command(str(path), str(lib)), check=True,
                   capture_output=True)
    o = oracle.Oracle(str(lib))
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(o)
        except (AssertionError, ValueError) as e:
            caught.append(pin.__name__)
            break
    assert caught, f"no pin catches the planted mistake '{name}'"
