"""Plant a mistake in a copy of the oracle and check that the pins catch it.

Each mutant is a one-line edit of q4_oracle.c (a plausible slip: a wrong
nibble order, a dropped term, a wrong sign or index, a transposed operand),
compiled on the CPU into a temporary library.  The pins must reject every
one of them; a mutant that passes all pins would mean the pins leave that
part of the oracle unchecked.
"""
import os

import pytest

import oracle as ora
from pins import ALL_PINS

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "q4_oracle.c")

MUTANTS = {
    "interleaved_nibbles": ("int q = (j < 16) ? (qs[j] & 0x0F) : (qs[j - 16] >> 4);",
                            "int q = (j % 2 == 0) ? (qs[j / 2] & 0x0F) : (qs[j / 2] >> 4);"),
    "swapped_nibbles": ("(qs[j] & 0x0F) : (qs[j - 16] >> 4)", "(qs[j] >> 4) : (qs[j - 16] & 0x0F)"),
    "no_offset": ("return (double)(q - 8) *", "return (double)(q) *"),
    "offset_7": ("return (double)(q - 8) *", "return (double)(q - 7) *"),
    "big_endian_scale": ("blk[0] | (blk[1] << 8)", "blk[1] | (blk[0] << 8)"),
    "flush_subnormals": ("v = ldexp((double)m, -24);", "v = 0.0;"),
    "exponent_bias": ("e - 25);", "e - 24);"),
    "ties_away": ("double m = rint(ldexp(a, 10 - e));", "double m = round(ldexp(a, 10 - e));"),
    "block_stride_16": ("#define ORA_BLOCK_BYTES 18", "#define ORA_BLOCK_BYTES 16"),
    "x_transposed": ("double p = ora_weight(w, k_dim, n, k) * ora_half_to_double(xb[k]);\n                acc += p;\n                mag += fabs(p);\n            }\n            y[(int64_t)b * n_rows + n] = acc;",
                     "double p = ora_weight(w, k_dim, n, k) * ora_half_to_double(x[k * batch + b]);\n                acc += p;\n                mag += fabs(p);\n            }\n            y[(int64_t)b * n_rows + n] = acc;"),
    "signed_magnitude": ("mag += fabs(p);", "mag += p;"),
    "attn_modulo": ("(qh / group) * head_dim", "(qh % n_kv) * head_dim"),
    "norm_no_mean": ("sqrt(ss / (double)dim + eps)", "sqrt(ss + eps)"),
    "add_sign": ("t[i] = ora_half_to_double(z[i]) + o[i];", "t[i] = ora_half_to_double(z[i]) - o[i];"),
    "layer_skips_norm": ("ora_add(z1, dn, (int64_t)batch * hidden, t2);\n    ora_rmsnorm_d(t2, batch, hidden, eps, z_out);",
                         "ora_add(z1, dn, (int64_t)batch * hidden, t2);\n    ora_double_to_half_n(t2, (int64_t)batch * hidden, z_out);"),
    "silu_sign": ("exp(-g[i])", "exp(g[i])"),
    "attn_scale": ("double scale = 1.0 / sqrt((double)head_dim);", "double scale = 1.0 / (double)head_dim;"),
    "attn_no_max_shift": ("work[t] = exp(work[t] - mx);", "work[t] = exp(work[t]);"),
    "attn_group_modulo": ("int64_t g = h / group;", "int64_t g = h % n_kv;"),
    "attn_cache_stride": ("kc[t * kv_dim + g * head_dim + i]", "kc[t * head_dim + g * head_dim + i]"),
    "attn_signed_sabs": ("aabs += work[t] / den * fabs(v);", "aabs += work[t] / den * v;"),
    "gate_up_swap": ("ora_silu_mul(g, u, (int64_t)batch * ffn, act);", "ora_silu_mul(u, g, (int64_t)batch * ffn, act);"),
    "attn_reads_k": ("ora_attn_ctx1(v, batch, q_dim, kv_dim, head_dim, attn);",
                     "ora_attn_ctx1(k, batch, q_dim, kv_dim, head_dim, attn);"),
    "o_reads_z": ("ora_gemv(wts[3], attn, hidden, q_dim, batch, 0, hidden, o, 0);",
                  "ora_gemv(wts[3], z, hidden, q_dim, batch, 0, hidden, o, 0);"),
    "down_reads_z1": ("ora_gemv(wts[6], act, hidden, ffn, batch, 0, hidden, dn, 0);",
                      "ora_gemv(wts[6], z1, hidden, ffn, batch, 0, hidden, dn, 0);"),
    "ffn_residual_base_z": ("ora_add(z1, dn, (int64_t)batch * hidden, t2);", "ora_add(z, dn, (int64_t)batch * hidden, t2);"),
    "attn_residual_base_dropped": ("ora_add(z, o, (int64_t)batch * hidden, t1);",
                                   "ora_add(z1, o, (int64_t)batch * hidden, t1);"),
    "k_weights_for_v": ("ora_gemv(wts[2], z, kv_dim, hidden, batch, 0, kv_dim, v, 0);",
                        "ora_gemv(wts[1], z, kv_dim, hidden, batch, 0, kv_dim, v, 0);"),
    "kv_row_off_by_one": ("ora_double_to_half_n(v, kv_dim, vc + pos * kv_dim);",
                          "ora_double_to_half_n(v, kv_dim, vc + (pos + 1) * kv_dim);"),
    "kv_context_excludes_token": ("ora_attn_decode(q, kc, vc, pos + 1, n_q, n_kv, head_dim, att, sabs, aw);",
                                  "ora_attn_decode(q, kc, vc, pos > 0 ? pos : 1, n_q, n_kv, head_dim, att, sabs, aw);"),
    "kv_k_into_v": ("ora_double_to_half_n(v, kv_dim, vc + pos * kv_dim);", "ora_double_to_half_n(k, kv_dim, vc + pos * kv_dim);"),
    "attn_value_key_swap": ("double v = ora_half_to_double(vc[t * kv_dim + g * head_dim + i]);",
                            "double v = ora_half_to_double(kc[t * kv_dim + g * head_dim + i]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site for {name} not found"
    src = tmp_path / f"mut_{name}.c"
    src.write_text(text.replace(old, new, 1))
    lib = ora.load(ora.compile_oracle(str(src), str(tmp_path / f"mut_{name}.so")))
    caught = []
    for pin in ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
        except Exception as e:  # a crash in a pin also rejects the mutant
            caught.append(f"{pin.__name__}:{type(e).__name__}")
    assert caught, f"mutant {name} passed every pin"
