"""Plant plausible mistakes in copies of the oracle (on the CPU) and check that
at least one pin catches each: the pins are chosen so that a dropped term, a
wrong sign or index, a transposed operand, a changed rounding order or a
misread choice of the pages fails one of them."""
import os

import pytest

import oracle
import test_oracle_brute as tb
import test_oracle_cell as tcell
import test_oracle_closed_form as tc
import test_oracle_hand as th
import test_oracle_invariants as ti
import test_oracle_math as tm

# (name, text in rnn_oracle.c, replacement)
MUTANTS = [
    ("k-descending dot", "for (long k = 0; k < K; ++k) acc = acc + x[k] * w[k];",
     "for (long k = K - 1; k >= 0; --k) acc = acc + x[k] * w[k];"),
    ("dot drops first term", "for (long k = 0; k < K; ++k) acc = acc + x[k] * w[k];",
     "for (long k = 1; k < K; ++k) acc = acc + x[k] * w[k];"),
    ("W index as [input, gates*hidden]", "xw[j] = o_dot(x, a->W + (d * GH + j) * a->I, a->I);",
     "{ float s = 0.0f; for (long k = 0; k < a->I; ++k) s = s + x[k] * a->W[d * GH * a->I + k * GH + j]; xw[j] = s; }"),
    ("RNN biases pre-summed", "if (a->B) { pre = pre + Wb[u]; pre = pre + Rb[u]; }",
     "if (a->B) { pre = pre + (Wb[u] + Rb[u]); }"),
    ("RNN drops Rb", "if (a->B) { pre = pre + Wb[u]; pre = pre + Rb[u]; }",
     "if (a->B) { pre = pre + Wb[u]; }"),
    ("GRU z/r swapped", "float pz = xw[u] + o_dot(h, Rd + u * H, H);",
     "float pz = xw[H + u] + o_dot(h, Rd + (H + u) * H, H);"),
    ("GRU update weights swapped", "hn[u] = (1.0f - z[u]) * ht + z[u] * h[u];",
     "hn[u] = z[u] * ht + (1.0f - z[u]) * h[u];"),
    ("GRU lbr0 without reset", "for (long k = 0; k < H; ++k) rh[k] = r[k] * h[k];",
     "for (long k = 0; k < H; ++k) rh[k] = h[k];"),
    ("GRU lbr1 biases exchanged", "ph = (xw[2 * H + u] + r[u] * (rec + Rb[2 * H + u])) + Wb[2 * H + u];",
     "ph = (xw[2 * H + u] + r[u] * (rec + Wb[2 * H + u])) + Rb[2 * H + u];"),
    ("LSTM o/f gates swapped", "float po = xw[H + u] + o_dot(h, Rd + (H + u) * H, H);",
     "float po = xw[2 * H + u] + o_dot(h, Rd + (2 * H + u) * H, H);"),
    ("LSTM Po with previous cell", "if (a->P) po = po + Po[u] * cn[u];",
     "if (a->P) po = po + Po[u] * c[u];"),
    ("LSTM drops Pf", "pf = pf + Pf[u] * c[u];", "pf = pf;"),
    ("LSTM cell terms crossed", "cn[u] = fg * c[u] + ig * ct;", "cn[u] = fg * ct + ig * c[u];"),
    ("input_forget uncoupled", "float fg = a->input_forget ? 1.0f - ig :", "float fg = a->input_forget ? ig :"),
    ("LSTM h uses g", "hn[u] = og * o_act(&acts[2], cn[u]);", "hn[u] = og * o_act(&acts[1], cn[u]);"),
    ("clip lower bound sign", "if (v < -a->clip) return -a->clip;", "if (v < -a->clip) return a->clip;"),
    ("clip 0 clamps", "a.has_clip = clip > 0.0f;", "a.has_clip = clip >= 0.0f;"),
    ("reverse ignores lens", "long t = reverse ? L - 1 - s : s;", "long t = reverse ? a->S - 1 - s : s;"),
    ("len-0 row returns initial state", "yh[u] = L > 0 ? o_canon(h[u]) : 0.0f;", "yh[u] = o_canon(h[u]);"),
    ("layout-1 Y index", "((n * a->S + t) * a->dirs + d) * a->H;", "((n * a->dirs + d) * a->S + t) * a->H;"),
    ("layout-1 X index", "(n * a->S + t) * a->I;", "(t * a->N + n) * a->I;"),
    ("beta shares the alpha cursor", "if (beta && cb < n_beta) list[i].beta = beta[cb];",
     "if (beta && ca - 1 < n_beta && ca > 0) list[i].beta = beta[ca - 1];"),
    ("second set ignored", "int base = (n_list == 2 * k && d == 1) ? k : 0;", "int base = 0;"),
    ("exp drops r^3 term", "p = p * r + E3;", "p = p * r;"),
    ("tanh large-range formula", "y = 1.0f - 2.0f / (e + 1.0f);", "y = 1.0f - 1.0f / (e + 1.0f);"),
    ("sigmoid sign", "return 1.0f / (1.0f + oracle_exp(-x));", "return 1.0f / (1.0f + oracle_exp(x));"),
    ("hardsigmoid upper clamp", "(v > 1.0f ? 1.0f : v)", "(v > 1.0f ? v : v)"),
    ("softplus threshold", "x > 20.0f ? x : oracle_log", "x > 2.0f ? x : oracle_log"),
    ("elu drops -1", "alpha * (oracle_exp(x) - 1.0f)", "alpha * oracle_exp(x)"),
    ("relu drops NaN", "case OA_RELU:            return x < 0.0f ? 0.0f : x;",
     "case OA_RELU:            return !(x >= 0.0f) ? 0.0f : x;"),
    ("NaN not canonical", "return o_isnan(x) ? o_from_bits(0x7FC00000u) : x;", "return x;"),
    ("leakyrelu default alpha", "case OA_LEAKYRELU: return 0.01f;", "case OA_LEAKYRELU: return 0.1f;"),
    ("cell drops B", "float pre = (xw + rec) + B[j];", "float pre = xw + rec;"),
    ("cell B added to rec first", "float pre = (xw + rec) + B[j];", "float pre = xw + (rec + B[j]);"),
    ("cell R transposed", "float rec = o_dot(Hprev + n * H, R + j * H, H);",
     "float rec = 0.0f; for (long k = 0; k < H; ++k) rec = rec + Hprev[n * H + k] * R[k * H + j];"),
    ("cell W and R exchanged", "float xw = o_dot(X + n * I, W + j * I, I);",
     "float xw = o_dot(X + n * I, R + j * I, I);"),
    ("cell clip lower bound sign", "else if (pre < -clip) pre = -clip;", "else if (pre < -clip) pre = clip;"),
    ("cell default sigmoid", "int fn = activation ? o_name_to_fn(activation) : OA_TANH;",
     "int fn = activation ? o_name_to_fn(activation) : OA_SIGMOID;"),
    ("cell accepts affine", "if (fn != OA_RELU && fn != OA_SIGMOID && fn != OA_TANH) return 1;",
     "if (fn < 0) return 1;"),
    ("LSTM drops Pi", "pi = pi + Pi[u] * c[u];", "pi = pi;"),
    ("LSTM Pf takes Pi", "pf = pf + Pf[u] * c[u];", "pf = pf + Pi[u] * c[u];"),
    ("LSTM cell state clipped", "hn[u] = og * o_act(&acts[2], cn[u]);",
     "hn[u] = og * o_act(&acts[2], o_clip(a, cn[u]));"),
    ("GRU lbr0 drops Rb", "if (a->B) { ph = ph + Wb[2 * H + u]; ph = ph + Rb[2 * H + u]; }",
     "if (a->B) { ph = ph + Wb[2 * H + u]; }"),
    ("thresholdedrelu boundary", "case OA_THRESHOLDEDRELU: return x > alpha ? x : 0.0f;",
     "case OA_THRESHOLDEDRELU: return x >= alpha ? x : 0.0f;"),
    ("scaledtanh alpha and beta swapped", "case OA_SCALEDTANH:      return alpha * oracle_tanh(beta * x);",
     "case OA_SCALEDTANH:      return beta * oracle_tanh(alpha * x);"),
    ("hardsigmoid lower clamp", "return v < 0.0f ? 0.0f : (v > 1.0f ? 1.0f : v);",
     "return v < 0.0f ? v : (v > 1.0f ? 1.0f : v);"),
    ("hardsigmoid default beta", "case OA_HARDSIGMOID: return 0.5f;", "case OA_HARDSIGMOID: return 0.0f;"),
    ("hardsigmoid default alpha", "case OA_HARDSIGMOID: return 0.2f;", "case OA_HARDSIGMOID: return 1.0f;"),
    ("softsign drops abs", "case OA_SOFTSIGN:        return x / (1.0f + o_fabs(x));",
     "case OA_SOFTSIGN:        return x / (1.0f + x);"),
    ("affine drops beta", "case OA_AFFINE:          return alpha * x + beta;",
     "case OA_AFFINE:          return alpha * x;"),
    ("scaledtanh takes no beta", "return fn == OA_AFFINE || fn == OA_SCALEDTANH || fn == OA_HARDSIGMOID;",
     "return fn == OA_AFFINE || fn == OA_HARDSIGMOID;"),
    ("GRU lbr0 reset by z", "for (long k = 0; k < H; ++k) rh[k] = r[k] * h[k];",
     "for (long k = 0; k < H; ++k) rh[k] = z[k] * h[k];"),
    ("GRU candidate takes f", "float ht = o_act(&acts[1], o_clip(a, ph));", "float ht = o_act(&acts[0], o_clip(a, ph));"),
    ("LSTM candidate takes f", "float ct = o_act(&acts[1], o_clip(a, pc));", "float ct = o_act(&acts[0], o_clip(a, pc));"),
    ("RNN takes g", "hn[u] = o_act(&acts[0], o_clip(a, pre));", "hn[u] = o_act(&acts[1], o_clip(a, pre));"),
    ("len-0 row returns initial cell", "for (long u = 0; u < H; ++u) yc[u] = L > 0 ? o_canon(c[u]) : 0.0f;",
     "for (long u = 0; u < H; ++u) yc[u] = o_canon(c[u]);"),
    ("dot starts from -0", "    float acc = 0.0f;\n    for (long k = 0; k < K; ++k) acc = acc + x[k] * w[k];",
     "    float acc = -0.0f;\n    for (long k = 0; k < K; ++k) acc = acc + x[k] * w[k];"),
    ("clip turns NaN into the bound", "    if (v > a->clip) return a->clip;", "    if (!(v <= a->clip)) return a->clip;"),
    ("clip before the peepholes", "                float ig = o_act(&acts[0], o_clip(a, pi));",
     "                float ig = o_act(&acts[0], o_clip(a, a->P ? pi - Pi[u] * c[u] : pi) + (a->P ? Pi[u] * c[u] : 0.0f));"),
    ("names case-sensitive", "            if (c >= 'A' && c <= 'Z') c = (char)(c - 'A' + 'a');\n", ""),
    ("elu default alpha", "    case OA_ELU: return 1.0f;", "    case OA_ELU: return 0.5f;"),
    ("thresholdedrelu default alpha", "    case OA_THRESHOLDEDRELU: return 1.0f;", "    case OA_THRESHOLDEDRELU: return 0.5f;"),
    ("scaledtanh default alpha", "    case OA_SCALEDTANH: return 1.0f;", "    case OA_SCALEDTANH: return 0.5f;"),
    ("affine default alpha", "    case OA_AFFINE: return 1.0f;", "    case OA_AFFINE: return 0.5f;"),
    ("affine default beta 1", "    default: return 0.0f;   /* Affine and ScaledTanh default beta is 0 */",
     "    default: return 1.0f;   /* Affine and ScaledTanh default beta is 0 */"),
    ("LSTM default h activation sigmoid", "list[1].fn = OA_TANH; list[2].fn = OA_TANH; }",
     "list[1].fn = OA_TANH; list[2].fn = OA_SIGMOID; }"),
    ("GRU default g activation sigmoid", "else if (op == 1) { list[0].fn = OA_SIGMOID; list[1].fn = OA_TANH; }",
     "else if (op == 1) { list[0].fn = OA_SIGMOID; list[1].fn = OA_SIGMOID; }"),
    ("Wb and Rb exchanged", "const float* Wb = a->B ? a->B + d * 2 * GH : NULL;\n    const float* Rb = a->B ? a->B + d * 2 * GH + GH : NULL;",
     "const float* Wb = a->B ? a->B + d * 2 * GH + GH : NULL;\n    const float* Rb = a->B ? a->B + d * 2 * GH : NULL;"),
    ("Po and Pf exchanged", "const float* Po = a->P ? a->P + d * 3 * H + H : NULL;\n    const float* Pf = a->P ? a->P + d * 3 * H + 2 * H : NULL;",
     "const float* Po = a->P ? a->P + d * 3 * H + 2 * H : NULL;\n    const float* Pf = a->P ? a->P + d * 3 * H + H : NULL;"),
    ("both directions start from direction 0's state", "h[u] = a->h0 ? a->h0[o_sidx(a, d, n) + u] : 0.0f;",
     "h[u] = a->h0 ? a->h0[o_sidx(a, 0, n) + u] : 0.0f;"),
    ("both directions use direction 0's R", "const float* Rd = a->R + d * GH * H;", "const float* Rd = a->R;"),
    ("layout-0 Y direction and batch axes exchanged", "return a->layout == 0 ? ((t * a->dirs + d) * a->N + n) * a->H",
     "return a->layout == 0 ? ((t * a->N + n) * a->dirs + d) * a->H"),
    ("layout-0 state direction and batch axes exchanged", "return a->layout == 0 ? (d * a->N + n) * a->H : (n * a->dirs + d) * a->H;",
     "return a->layout == 0 ? (n * a->dirs + d) * a->H : (n * a->dirs + d) * a->H;"),
    ("bidirectional second direction forward", "int reverse = direction == 1 || (direction == 2 && d == 1);",
     "int reverse = direction == 1;"),
    ("GRU lbr1 without B resets xw too", "else ph = xw[2 * H + u] + r[u] * rec;", "else ph = r[u] * (xw[2 * H + u] + rec);"),
    ("GRU lbr0 Wb inside the reset", "ph = xw[2 * H + u] + o_dot(rh, Rh, H);\n                    if (a->B) { ph = ph + Wb[2 * H + u]; ph = ph + Rb[2 * H + u]; }",
     "ph = xw[2 * H + u] + o_dot(rh, Rh, H);\n                    if (a->B) { ph = ph + r[u] * Wb[2 * H + u]; ph = ph + Rb[2 * H + u]; }"),
    ("cell accepts clip 0", "if (!(clip > 0.0f)) return 1;", "if (clip < 0.0f) return 1;"),
    ("cell clips NaN to the bound", "            if (pre > clip) pre = clip;", "            if (!(pre <= clip)) pre = clip;"),
    ("cell batch rows share Hprev", "float rec = o_dot(Hprev + n * H, R + j * H, H);", "float rec = o_dot(Hprev, R + j * H, H);"),
    ("cell NaN not canonical", "Ho[n * H + j] = o_canon(oracle_activation(fn, 0.0f, 0.0f, pre));",
     "Ho[n * H + j] = oracle_activation(fn, 0.0f, 0.0f, pre);"),
    ("LSTM Rb before Wb", "pi = pi + Wb[u];         pi = pi + Rb[u];", "pi = pi + Rb[u];         pi = pi + Wb[u];"),
    ("GRU Rb before Wb", "pz = pz + Wb[u]; pz = pz + Rb[u];", "pz = pz + Rb[u]; pz = pz + Wb[u];"),
    ("LSTM bias before rec", "float pc = xw[3 * H + u] + o_dot(h, Rd + (3 * H + u) * H, H);",
     "float pc = (a->B ? xw[3 * H + u] + Wb[3 * H + u] : xw[3 * H + u]) + o_dot(h, Rd + (3 * H + u) * H, H);"),
    ("GRU lbr0 candidate Rb before Wb", "if (a->B) { ph = ph + Wb[2 * H + u]; ph = ph + Rb[2 * H + u]; }",
     "if (a->B) { ph = ph + Rb[2 * H + u]; ph = ph + Wb[2 * H + u]; }"),
    ("GRU update as ht + z*(h - ht)", "hn[u] = (1.0f - z[u]) * ht + z[u] * h[u];", "hn[u] = ht + z[u] * (h[u] - ht);"),
    ("LSTM peephole before the biases",
     "                if (a->B) {\n"
     "                    pi = pi + Wb[u];         pi = pi + Rb[u];\n"
     "                    po = po + Wb[H + u];     po = po + Rb[H + u];\n"
     "                    pf = pf + Wb[2 * H + u]; pf = pf + Rb[2 * H + u];\n"
     "                    pc = pc + Wb[3 * H + u]; pc = pc + Rb[3 * H + u];\n"
     "                }\n"
     "                if (a->P) {\n"
     "                    pi = pi + Pi[u] * c[u];\n"
     "                    pf = pf + Pf[u] * c[u];\n"
     "                }\n",
     "                if (a->P) {\n"
     "                    pi = pi + Pi[u] * c[u];\n"
     "                    pf = pf + Pf[u] * c[u];\n"
     "                }\n"
     "                if (a->B) {\n"
     "                    pi = pi + Wb[u];         pi = pi + Rb[u];\n"
     "                    po = po + Wb[H + u];     po = po + Rb[H + u];\n"
     "                    pf = pf + Wb[2 * H + u]; pf = pf + Rb[2 * H + u];\n"
     "                    pc = pc + Wb[3 * H + u]; pc = pc + Rb[3 * H + u];\n"
     "                }\n"),
    ("elu at -0 takes the exp branch", "case OA_ELU:             return x >= 0.0f ? x : alpha * (oracle_exp(x) - 1.0f);",
     "case OA_ELU:             return x > 0.0f ? x : alpha * (oracle_exp(x) - 1.0f);"),
    ("relu turns -0 into +0", "case OA_RELU:            return x < 0.0f ? 0.0f : x;", "case OA_RELU:            return x <= 0.0f ? 0.0f : x;"),
    ("hardsigmoid drops NaN", "return v < 0.0f ? 0.0f : (v > 1.0f ? 1.0f : v);", "return !(v >= 0.0f) ? 0.0f : (v > 1.0f ? 1.0f : v);"),
    ("softplus drops the 1", "x > 20.0f ? x : oracle_log(1.0f + oracle_exp(x))", "x > 20.0f ? x : oracle_log(oracle_exp(x))"),
    ("leakyrelu NaN to 0", "case OA_LEAKYRELU:       return x < 0.0f ? alpha * x : x;", "case OA_LEAKYRELU:       return x >= 0.0f ? x : alpha * (x != x ? 0.0f : x);"),
    ("reverse Y written in step order", "            float* y = a->Y + o_yidx(a, t, d, n);\n            for (long u = 0; u < H; ++u) y[u] = o_canon(h[u]);",
     "            float* y = a->Y + o_yidx(a, s, d, n);\n            for (long u = 0; u < H; ++u) y[u] = o_canon(h[u]);"),
    ("layout-0 X index batch-major", "return a->layout == 0 ? (t * a->N + n) * a->I : (n * a->S + t) * a->I;",
     "return a->layout == 0 ? (n * a->S + t) * a->I : (n * a->S + t) * a->I;"),
    ("reverse projects step s", "        o_project(a, d, t, n, xw);", "        o_project(a, d, s, n, xw);"),
    ("exp overflow threshold 88", "if (x > 89.0f) return o_from_bits(0x7F800000u);",
     "if (x > 88.0f) return o_from_bits(0x7F800000u);"),
    ("exp underflow threshold -100", "if (x < -110.0f) return 0.0f;", "if (x < -100.0f) return 0.0f;"),
    ("exp drops the ln2 tail", "float r = (x - kf * LN2_HEAD) - kf * LN2_TAIL;", "float r = x - kf * LN2_HEAD;"),
    ("log subnormal exponent", "        eadj = -24;", "        eadj = -23;"),
    ("tanh loses the sign", "    return o_from_bits(o_to_bits(y) | sign);", "    return y;"),
    ("tanh saturates early", "if (a > 9.1f) {", "if (a > 5.0f) {"),
    ("alpha cursor advances without a taker", "            if (o_takes_alpha(fn)) {\n                if (alpha && ca < n_alpha) list[i].alpha = alpha[ca];\n                ca++;\n            }",
     "            if (o_takes_alpha(fn)) {\n                if (alpha && ca < n_alpha) list[i].alpha = alpha[ca];\n            }\n            ca++;"),
]


def _battery():
    """Run the pins; return the names of those that fail."""
    checks = []
    for p in th.FILES:
        checks.append((f"golden {os.path.basename(p)}", lambda p=p: th.test_golden_case(p)))
    checks.append(("nan canonical", th.test_nan_outputs_are_canonical))
    checks.append(("plus zero start", th.test_accumulation_starts_from_plus_zero))
    checks.append(("nan through clip", th.test_nan_passes_through_clip))
    checks.append(("bidi lens hand", th.test_bidirectional_lens_combines_both_hand_cases))
    for s in range(25):
        checks.append((f"brute {s}", lambda s=s: tb.test_oracle_matches_float64_brute_force(s)))
    checks.append(("closed form", lambda: tc.test_affine_rnn_matches_integer_closed_form(0)))
    checks.append(("closed form reverse", tc.test_reverse_affine_closed_form))
    for s in range(3):
        checks.append((f"reverse {s}", lambda s=s: ti.test_reverse_is_forward_on_flipped_rows(s)))
        checks.append((f"bidi {s}", lambda s=s: ti.test_bidirectional_is_two_directions(s)))
        checks.append((f"layout {s}", lambda s=s: ti.test_layout1_is_transposed_layout0(s)))
        checks.append((f"lens {s}", lambda s=s: ti.test_sequence_lens_semantics(s)))
    checks.append(("resolve page case", ti.test_resolve_page_black_box_case))
    checks.append(("resolve workload", ti.test_resolve_lstm_bidi_workload))
    checks.append(("resolve defaults", ti.test_resolve_defaults_and_case_and_single_set))
    checks.append(("resolve page defaults", ti.test_resolve_every_default_the_page_lists))
    checks.append(("invalid lengths", ti.test_invalid_lengths_and_arguments))
    checks.append(("rnncell3", lambda: ti.test_rnncell3_one_step("tanh")))
    checks.append(("bnns gru", ti.test_bnns_gru_reset_after_matmul))
    for p in tcell.FILES:
        checks.append((f"cell golden {os.path.basename(p)}", lambda p=p: tcell.test_cell_golden(p)))
    for s in range(6):
        checks.append((f"cell float64 {s}", lambda s=s: tcell.test_cell_matches_float64(s)))
    checks.append(("cell defaults", tcell.test_cell_default_activation_is_tanh_and_default_clip_clamps_nothing))
    for act in tcell.ACTS:
        for clip in (None, 0.25):
            checks.append((f"cell sequence {act} {clip}",
                           lambda a=act, c=clip: tcell.test_cell_is_the_sequence_operator_at_one_step(a, c)))
    checks.append(("cell clip", tcell.test_cell_clip_saturates_exactly))
    checks.append(("cell nan", tcell.test_cell_nan_is_canonical))
    for bad in (dict(activation="Affine"), dict(clip=0.0), dict(clip=-1.0), dict(clip=float("nan"))):
        checks.append((f"cell rejects {bad}", lambda b=bad: tcell.test_cell_rejects_what_the_page_excludes(b)))
    for fn in (tm.test_exp_special_values, tm.test_log_special_values, tm.test_tanh_special_values,
               tm.test_relu_points, tm.test_leaky_thresholded_points,
               tm.test_hardsigmoid_affine_softsign_points, tm.test_softplus_points,
               tm.test_elu_scaledtanh_points):
        checks.append((fn.__name__, fn))
    checks.append(("exp sweep", tm.test_exp_accuracy_sweep))
    checks.append(("log sweep", tm.test_log_accuracy_sweep))
    checks.append(("sigmoid sweep", tm.test_sigmoid_accuracy_sweep))
    checks.append(("tanh sweep", tm.test_tanh_accuracy_sweep))
    checks.append(("softplus elu sweep", tm.test_softplus_elu_softsign_sweeps))
    failed = []
    for name, fn in checks:
        try:
            fn()
        except (Exception, pytest.fail.Exception):     # pytest.raises reports through the latter
            failed.append(name)
    return failed


def test_unmutated_oracle_passes_battery():
    assert _battery() == []


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    src = oracle.source()
    assert src.count(old) == 1, f"mutation anchor not unique/present: {old!r}"
    lib = oracle.compile_variant(src.replace(old, new), str(tmp_path / "mutant.so"))
    with oracle.use_library(lib):
        failed = _battery()
    assert failed, f"no pin caught the planted mistake: {name}"
