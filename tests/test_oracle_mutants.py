"""Planted mistakes in the oracle must be caught by its pins (CPU only).

Each mutant is a one-line edit of a copy of oracle/clo_oracle.c (a dropped
term, a wrong sign, index or operand).  The copy is compiled with gcc and the
full pin set is run on it in a child process; the test passes when at least
one pin fails for every mutant.  The real oracle source is never modified.
"""
import concurrent.futures as cf
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

MUTANTS = [
    ("Eq. 9 sign", "(1.0 - lam) * M_PI", "(1.0 + lam) * M_PI"),
    ("Eq. 7 arccos", "double theta_star = acos(eta);", "double theta_star = cos(eta);"),
    ("Eq. 8 power", "double lam = pow(sg, n_exp);", "double lam = sg * n_exp;"),
    ("group mean dropped", "sg /= (double)group;", ""),
    ("cosine normalisation", "return ab / (sqrt(aa) * sqrt(bb));", "return ab / (aa * bb);"),
    ("cosine operand", "aa += x * x;", "aa += x * y;"),
    ("Eq. 10 weight dropped", "swc += w_q[h] * c;", "swc += c;"),
    ("tie is a miss", "} else if (s >= tau_kv[g]) {", "} else if (s > tau_kv[g]) {"),
    ("strided GQA grouping", "int h = g * G + j;", "int h = j * Hkv + g;"),
    ("label not replaced",
     "memcpy(labels + off, q + off, (size_t)d * sizeof(uint16_t));", ""),
    ("miss list order", "miss_list[nmiss++] = b * Hkv + g;", "miss_list[nmiss++] = g * B + b;"),
    ("persistent ignored", "if (persist && persist[g]) {", "if (0) {"),
    ("scale dropped", "sc[t] = dot * scale;", "sc[t] = dot;"),
    ("lse max dropped", "lse[h] = m + log(l);", "lse[h] = log(l);"),
    ("normalisation dropped", "out[(size_t)h * d + i] = acc[i] / l;", "out[(size_t)h * d + i] = acc[i];"),
    ("softmax shift sign", "double p = exp(sc[t] - m);", "double p = exp(sc[t] + m);"),
    ("index ignored", "int r = rows ? rows[t] : t;", "int r = t;"),
    ("persist slot by position", "if (persist_ids[j] == g) slot = j;", "if (j == g) slot = j;"),
    ("persistent batch/slot swap", "size_t base = (((size_t)b * Np + slot) * (size_t)T) * d;",
     "size_t base = (((size_t)slot * B + b) * (size_t)T) * d;"),
    ("paged row in block", "h) * block_size + t % block_size) * d;",
     "h) * block_size + t / block_size) * d;"),
    ("paged GQA query offset", "size_t qo = ((size_t)r * Hq + (size_t)h * G) * d;",
     "size_t qo = ((size_t)r * Hq + (size_t)h) * d;"),
    ("binary16 exponent bias", "v = ldexp((double)(1024 + m), e - 25);",
     "v = ldexp((double)(1024 + m), e - 24);"),
    ("binary16 subnormal scale", "v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    ("fill slot ignored", "int r = slot ? slot[sel] : t;", "int r = t;"),
    ("fill K from V", "memcpy(cbK + to, srcK + from,", "memcpy(cbK + to, srcV + from,"),
    ("fill miss list ignored", "int e = miss_list[m];", "int e = m;"),
    ("fill source row by position", "size_t from = ((size_t)e * T + t) * d;",
     "size_t from = ((size_t)e * T + j) * d;"),
    ("Eq. 11 margin sign", "D[at] = tau[at] - (s_hat[at] - eps);",
     "D[at] = tau[at] - (s_hat[at] + eps);"),
    ("Eq. 12 as printed", "double cap = floor(t_comp * b_link / mem_head);",
     "double cap = floor(t_comp / (b_link * mem_head));"),
    ("Eq. 13 clamp dropped", "if (keep < 0) keep = 0;", ""),
    ("hard at zero difficulty", "if (D[at] > 0) ++hard;", "if (D[at] >= 0) ++hard;"),
    ("easiest heads kept", "if (best < 0 || D[at] > D[(size_t)l * Hkv + best]) best = i;",
     "if (best < 0 || D[at] < D[(size_t)l * Hkv + best]) best = i;"),
    ("tie goes to the higher head", "if (best < 0 || D[at] > D[(size_t)l * Hkv + best]) best = i;",
     "if (best < 0 || D[at] >= D[(size_t)l * Hkv + best]) best = i;"),
    ("top-k one query of the group", "acc += oracle_half_to_double(q[((size_t)b * Hq + (size_t)g * G + j) * d + i]);",
     "acc += oracle_half_to_double(q[((size_t)b * Hq + (size_t)g * G) * d + i]);"),
    ("top-k strided grouping", "acc += oracle_half_to_double(q[((size_t)b * Hq + (size_t)g * G + j) * d + i]);",
     "acc += oracle_half_to_double(q[((size_t)b * Hq + (size_t)j * Hkv + g) * d + i]);"),
    ("top-k smallest scores", "if (si > sj) return -1;", "if (si < sj) return -1;"),
    ("top-k ties to higher token", "return i < j ? -1 : (i > j);", "return i > j ? -1 : (i < j);"),
    ("top-k output not ascending", "qsort(order, (size_t)k, sizeof(int), by_index);", ""),
    ("fill last row dropped", "for (int j = 0; j < k; ++j) {\n            size_t sel",
     "for (int j = 0; j < k - 1; ++j) {\n            size_t sel"),
]

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

CHILD = (
    "import sys; sys.path[:0] = [{root!r}, {tests!r}];"
    "import oracle, oracle_pins;"
    "failed = oracle_pins.run_all(oracle.Oracle({lib!r}));"
    "print(len(failed), failed[:1]);"
    "sys.exit(0 if failed else 17)"
)


def _run_mutant(tmpdir, i, old, new):
    src = open(oracle.SOURCE).read()
    assert src.count(old) == 1, f"mutant anchor not unique in oracle source: {old!r}"
    path_c = os.path.join(tmpdir, f"m{i}.c")
    path_so = os.path.join(tmpdir, f"m{i}.so")
    with open(path_c, "w") as f:
        f.write(src.replace(old, new))
    oracle.build(path_c, path_so)
    code = CHILD.format(root=ROOT, tests=HERE, lib=path_so)
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=300)
    return p.returncode, p.stdout + p.stderr[-500:]


def test_every_planted_mistake_is_caught():
    with tempfile.TemporaryDirectory() as tmp:
        with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            futs = {ex.submit(_run_mutant, tmp, i, o, n): name
                    for i, (name, o, n) in enumerate(MUTANTS)}
            survivors = []
            for fut in cf.as_completed(futs):
                rc, out = fut.result()
                # rc 0: some pin failed; a crash (negative rc) also counts as caught.
                if rc == 17:
                    survivors.append(futs[fut])
    assert not survivors, f"mutants not caught by any pin: {survivors}"
