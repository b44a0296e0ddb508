"""Planted mistakes in the oracle must each fail at least one pin.

Every mutation below is a plausible slip (a swapped operand, a dropped term,
a wrong index, sign or tag) applied to a copy of oracle/isd_oracle.c, built
on the CPU into a temporary library.  The pins of tests/oracle_pins.py run on
that build; a mutation that no pin catches fails this test.
"""
import os
import subprocess

import pytest

import oracle
import oracle_pins

SOURCE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "oracle", "isd_oracle.c")

MUTATIONS = {
    "ratio p/q swapped": ("double r = exp(lp - lq);", "double r = exp(lq - lp);"),
    "min(1, .) dropped": ("return r < 1.0 ? r : 1.0;", "return r;"),
    "residual sign": ("double d = pp[v] - qq[v];", "double d = qq[v] - pp[v];"),
    "residual fallback dropped": ("if (total == 0.0)\n", "if (0)\n"),
    "icdf boundary": ("if (c > t) { chosen = v; break; }", "if (c >= t) { chosen = v; break; }"),
    "icdf unscaled target": ("double t = u * S;", "double t = u;"),
    "accept test reversed": ("accepted = u_accept[k - 1] < racc;",
                             "accepted = u_accept[k - 1] > racc;"),
    "relaxation divides": ("fmin(1.0, (1.0 + tau) * exp(log_px - log_qx))",
                           "fmin(1.0, exp(log_px - log_qx) / (1.0 + tau))"),
    "relaxed ratio reported": ("        if (tau != 0.0)\n            racc", "        if (tau != 0.0)\n            ratio[k - 1] = racc"),
    "prefix not stopped": ("if (!accepted) break;", "if (!accepted) continue;"),
    "top-k keeps one more": ("int kept = (top_k > 0 && top_k < V) ? top_k : V;",
                             "int kept = (top_k > 0 && top_k < V) ? top_k + 1 : V;"),
    "filter ties to higher id": ("return x->id - y->id;", "return y->id - x->id;"),
    "filtered not renormalised": ("out[r[j].id] = r[j].p / total;", "out[r[j].id] = r[j].p;"),
    "top-p over the whole row": ("cum += r[j].p / sk;", "cum += r[j].p;"),
    "greedy accepts all": ("accepted = ratio[k - 1] == 1.0;", "accepted = 1;"),
    "alpha denominator": ("*alpha = sum / L;", "*alpha = sum / (L + 1);"),
    "bonus row": ("const double* Pb = P + (size_t)L * V;",
                  "const double* Pb = P + (size_t)(L - 1) * V;"),
    "correction row": ("const double* Pj = P + (size_t)(j - 1) * V;",
                       "const double* Pj = P + (size_t)j * V;"),
    "argmax tie to highest": ("if (logits[v] > logits[best]) best = v;",
                              "if (logits[v] >= logits[best]) best = v;"),
    "q not tempered": ("double lq = oracle_log_softmax_at(Q, V, T, x);",
                       "double lq = oracle_log_softmax_at(Q, V, 1.0, x);"),
    "softmax not tempered": ("out[v] = exp(logits[v] / T - zmax);", "out[v] = exp(logits[v] - zmax);"),
    "log-partition sign": ("return logits[x] / T - zmax - log(total);",
                           "return logits[x] / T - zmax + log(total);"),
    "correction reuses accept draw": (
        "u_cor[k - 1] = oracle_uniform(seed, offset, (uint64_t)i, (uint64_t)k, TAG_CORRECT);",
        "u_cor[k - 1] = oracle_uniform(seed, offset, (uint64_t)i, (uint64_t)k, TAG_ACCEPT);"),
    "bonus reuses last accept draw": ("(uint64_t)(L + 1), TAG_BONUS);", "(uint64_t)L, TAG_ACCEPT);"),
    "propose reuses accept draw": ("(uint64_t)m, TAG_PROPOSE);", "(uint64_t)m, TAG_ACCEPT);"),
    "philox multiplier": ("M0 = 0xD2E7470EE14C6C93ULL", "M0 = 0xD2E7470EE14C6C95ULL"),
    "philox key schedule": ("if (round > 0) { k0 += W0; k1 += W1; }", "if (round > 1) { k0 += W0; k1 += W1; }"),
    "uniform bits": ("return (double)(out[0] >> 40) * (1.0 / 16777216.0);",
                     "return (double)(out[0] >> 41) * (1.0 / 16777216.0);"),
    "anchor rows not shifted": ("load_rows(p_logits, dtype, ld_p, (int64_t)start + i, L + 1, V, P);",
                                "load_rows(p_logits, dtype, ld_p, (int64_t)start, L + 1, V, P);"),
    "kv keeps no x_last": ("*kept = 1 + a;", "*kept = a;"),
    "kv verifies after a rejection": ("*next_pend = (L == 0 || a == L) ? M : 0;", "*next_pend = M;"),
    "kv reads accept of proposal-only": ("int a = L > 0 ? a_in : 0;", "int a = a_in;"),
    "kv trimmed entry not cleared": ("            *e = -1;\n", ""),
    "kv block from stack bottom": ("int64_t next = top - wanted;", "int64_t next = 0;"),
    "kv pool check off by one": ("if (top + pushed < wanted) return KV_ERR_POOL;",
                                 "if (top + pushed <= wanted) return KV_ERR_POOL;"),
    "kv capacity off by one": ("+ 1 + *next_pend + M > ld)", "+ 1 + *next_pend + M >= ld)"),
    "kv slot range": ("slot >= pool_size", "slot > pool_size"),
    "kv allocation after the trimmed": ("int len = seq_len[i] + kept;", "int len = seq_len[i] + alloc[i];"),
    "gumbel noise sign": ("double score = log(w[v]) - log(-log(u));", "double score = log(w[v]) + log(-log(u));"),
    "gumbel ignores the weights": ("double score = log(w[v]) - log(-log(u));", "double score = -log(-log(u));"),
    "gumbel weights not logged": ("double score = log(w[v]) - log(-log(u));", "double score = w[v] - log(-log(u));"),
    "gumbel uniform word": ("out[v % GUMBEL_IDS_PER_BLOCK] >> 41", "out[0] >> 41"),
    "gumbel block index": ("256 * (v / GUMBEL_IDS_PER_BLOCK)", "256 * v"),
    "bf16 decoding": ("uint32_t bits = (uint32_t)h << 16;", "uint32_t bits = (uint32_t)h << 15;"),
}


@pytest.fixture(scope="module")
def source():
    with open(SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_mutation_is_caught(name, source, tmp_path):
    old, new = MUTATIONS[name]
    assert source.count(old) == 1, f"mutation site not unique: {old!r}"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", "-fvisibility=hidden",
                    str(src), "-o", str(lib), "-lm"], check=True)
    mutant = oracle.Oracle(str(lib))
    caught = None
    for pin in oracle_pins.ALL_PINS:  # the first pin that fails is enough
        try:
            pin(mutant)
        except AssertionError:
            caught = pin.__name__
            break
    assert caught, f"no pin catches the mutation {name!r}"
