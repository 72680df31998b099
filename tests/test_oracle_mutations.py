"""The oracle's pins catch plausible mistakes in the oracle itself.

Each case plants one mistake in a copy of oracle/a2ats_oracle.c (a dropped
term, a wrong sign, a transposed index, an off-by-one, a wrong tie rule),
builds it with the oracle's own compile step, and runs the pin tests of the
routine it touches against that library (A2ATS_ORACLE_LIB, in a child
pytest): at least one pin must fail.  The Python-level routines (the step's
composition, the split size, the byte accounting) get the same treatment
through a planted copy of the oracle package placed first on the child's
path.  CPU only; nothing here touches the CUDA library.
"""
import os
import shutil
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

# name, text in the oracle source, planted text, pin files that must catch it
MUTATIONS = [
    ("rope sign", "y[a] = xa * c - xb * s;", "y[a] = xa * c + xb * s;", ["rope"]),
    ("rope frequency", "pow(base, -2.0 * (double)i / (double)d)",
     "pow(base, -(double)i / (double)d)", ["rope"]),
    ("window boundary off by one", "dist < window;\n        double pos",
     "dist <= window;\n        double pos", ["rope"]),
    ("second moment not averaged", "(M > 0 ? s / (double)M : 0.0)", "(M > 0 ? s : 0.0)",
     ["calib"]),
    ("ridge off the diagonal too", "(a == b ? ridge : 0.0)", "ridge", ["calib"]),
    ("cholesky index transposed", "s -= l[i * d + k] * l[j * d + k];",
     "s -= l[i * d + k] * l[k * d + j];", ["calib"]),
    ("quadratic form drops a factor", "v += diff[a] * row;", "v += row;", ["assign"]),
    ("row times L transposed", "s += v[a] * l[a * d + b];", "s += v[a] * l[b * d + a];",
     ["assign", "kmeans"]),
    ("ties to the highest index", "if (v < *b1) { *b2 = *b1;", "if (v <= *b1) { *b2 = *b1;",
     ["assign"]),
    ("blend weights swapped", "double s = -p->beta * err + (1.0 - p->beta) * cosv;",
     "double s = -(1.0 - p->beta) * err + p->beta * cosv;", ["assign"]),
    ("blend error not normalised", "double err = m > 0.0 ? e[j] / m : 0.0;",
     "double err = e[j];", ["assign"]),
    ("split cosine without the query norm",
     "double v = (kn > 0.0 && qn > 0.0) ? dot / (kn * qn) : 0.0;",
     "double v = (kn > 0.0 && qn > 0.0) ? dot / kn : 0.0;", ["split"]),
    ("split ties to the higher index", "return (x->i > y->i) - (x->i < y->i);",
     "return (x->i < y->i) - (x->i > y->i);", ["split", "attention"]),
    ("far query rotated the wrong way", "orc_rope_row(q, qf, d, far_b, base, interleaved);",
     "orc_rope_row(q, qf, d, -far_b, base, interleaved);", ["attention"]),
    ("near key rotated at the distance",
     "orc_rope_row(keys + j * d, kr, d, (double)j, base, interleaved);",
     "orc_rope_row(keys + j * d, kr, d, (double)(t - j), base, interleaved);", ["attention"]),
    ("out-of-range code reads centroid 0", "? codebook[(int64_t)c * d + a] : 0.0;",
     "? codebook[(int64_t)c * d + a] : codebook[a];", ["dequant"]),
    ("back substitution sign", "s -= ci[a] * l[a * d + b];", "s += ci[a] * l[a * d + b];",
     ["kmeans"]),
    ("first centre ignores its draw", "int64_t first = (int64_t)floor(u[0] * (double)n);",
     "int64_t first = 0;", ["kmeans"]),
    ("draw not scaled by the D^2 sum", "double target = u[k] * total, run = 0.0;",
     "double target = u[k], run = 0.0;", ["kmeans"]),
    ("mean over one member too many", "sum[j * d + a] / (double)cnt[j];",
     "sum[j * d + a] / (double)(cnt[j] + 1);", ["kmeans"]),
    ("empty centre moved", "if (cnt[j] > 0)\n", "if (1)\n", ["kmeans"]),
    ("second best kept wrong", "else if (v < *b2) { *b2 = v; }",
     "else if (v > *b2) { *b2 = v; }", ["assign"]),
    ("threshold score of the split off by rank",
     "if (kth) *kth = count > 0 ? s[count - 1].s : INFINITY;\n    qsort(perm, (size_t)count, "
     "sizeof(int32_t), by_value);\n    qsort(perm + count, (size_t)(n - count), "
     "sizeof(int32_t), by_value);\n    free(s);\n    return count;\n}\n\n/* ----",
     "if (kth) *kth = count > 0 ? s[0].s : INFINITY;\n    qsort(perm, (size_t)count, "
     "sizeof(int32_t), by_value);\n    qsort(perm + count, (size_t)(n - count), "
     "sizeof(int32_t), by_value);\n    free(s);\n    return count;\n}\n\n/* ----", ["split"]),
    ("split size rounded down",
     "if (scores) scores[i] = v;\n    }\n    int64_t count = (int64_t)ceil(",
     "if (scores) scores[i] = v;\n    }\n    int64_t count = (int64_t)floor(", ["split"]),
    ("retrieved count rounded down",
     "if (scores) scores[j] = u;\n    }\n    int64_t count = (int64_t)ceil(",
     "if (scores) scores[j] = u;\n    }\n    int64_t count = (int64_t)floor(", ["attention"]),
    ("blend cosine unnormalised", "cosv = dot / (qn * p->cnorm[j]);", "cosv = dot;",
     ["assign"]),
    ("far offset ignored", "double pos = near ? (double)p[r] : far_offset;",
     "double pos = near ? (double)p[r] : 0.0;", ["rope"]),
    ("attention window edge off by one",
     "int near = window > 0 && dist >= 0 && dist < window;\n        double u = 0.0;",
     "int near = window > 0 && dist >= 0 && dist <= window;\n        double u = 0.0;",
     ["attention"]),
    ("cholesky square root dropped", "l[i * d + i] = sqrt(s);", "l[i * d + i] = s;",
     ["calib"]),
    ("cholesky failing minor off by one", "if (!(s > 0.0)) return (int)(i + 1);",
     "if (!(s > 0.0)) return (int)i;", ["calib"]),
    ("blend beta = 1 not reduced exactly", "if (p->beta == 1.0) {", "if (p->beta == 2.0) {",
     ["assign"]),
    ("final objective dropped",
     "objective[iters] = assign_all(z, n, d, centroids, K, codes);",
     "objective[iters] = 0.0;", ["kmeans"]),
    ("k-means distance not squared", "double t = a[i] - b[i];\n        s += t * t;",
     "double t = a[i] - b[i];\n        s += fabs(t);", ["kmeans"]),
    ("z-space distance not squared",
     "for (int64_t b = 0; b < d; b++) { double e = z[b] - cj[b]; v += e * e; }",
     "for (int64_t b = 0; b < d; b++) { double e = z[b] - cj[b]; v += fabs(e); }",
     ["assign"]),
]


@pytest.mark.parametrize("name,old,new,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, pins, tmp_path):
    with open(os.path.join(ROOT, "oracle", "a2ats_oracle.c")) as f:
        src = f.read()
    assert src.count(old) == 1, f"the text to change must occur once: {old!r}"
    planted = tmp_path / "planted.c"
    planted.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(planted), str(tmp_path / "planted.so"))
    files = [os.path.join(HERE, f"test_oracle_{p}.py") for p in pins]
    env = dict(os.environ, A2ATS_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *files], cwd=ROOT, env=env, capture_output=True, text=True)
    assert r.returncode == 1, f"{name}: no pin failed\n{r.stdout[-2000:]}"


# planted mistakes in the Python composition of oracle/__init__.py
PY_MUTATIONS = [
    ("retrieval rows take the plain rule",
     "cr, a, b = assign_cholesky(kt[ret], c, l, nthreads)",
     "cr, a, b = assign_cholesky(kt[ret], c, None, nthreads)", ["pipeline"]),
    ("bulk rows take the H rule", "cb, a, b = assign_cholesky(kt[bulk], c, None, nthreads)",
     "cb, a, b = assign_cholesky(kt[bulk], c, l, nthreads)", ["pipeline"]),
    ("proxy query from the first row", "    q = kt[t]\n", "    q = kt[0]\n", ["pipeline"]),
    ("blend with each row as its own query",
     "cr, a, b = assign_blend(kt[ret], c, q, beta, nthreads)",
     "cr, a, b = assign_blend(kt[ret], c, kt[ret], beta, nthreads)", ["pipeline"]),
    ("far offset dropped in the step",
     "kt = windowed_rope(k, pos, t, window, far_offset, base, interleaved)",
     "kt = windowed_rope(k, pos, t, window, 0, base, interleaved)", ["pipeline"]),
    ("split size rounded down", "return min(n, max(0, math.ceil(float(fraction) * n)))",
     "return min(n, max(0, math.floor(float(fraction) * n)))", ["split"]),
    ("value bytes dropped", "    cv, fv = ck, fk\n", "    cv, fv = 0.0, fk\n", ["dequant"]),
    ("codebook bytes per bit", '"codebook_bytes": float((1 << codebook_bits) * sub_dim * 2)',
     '"codebook_bytes": float(codebook_bits * sub_dim * 2)', ["dequant"]),
]


@pytest.mark.parametrize("name,old,new,pins", PY_MUTATIONS, ids=[m[0] for m in PY_MUTATIONS])
def test_planted_python_mistake_is_caught(name, old, new, pins, tmp_path):
    pkg = os.path.join(ROOT, "oracle")
    with open(os.path.join(pkg, "__init__.py")) as f:
        src = f.read()
    assert src.count(old) == 1, f"the text to change must occur once: {old!r}"
    shutil.copytree(pkg, tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("*.so", "*.tmp*", "__pycache__"))
    (tmp_path / "oracle" / "__init__.py").write_text(src.replace(old, new))
    env = dict(os.environ, A2ATS_ORACLE_LIB=oracle.build(),
               PYTHONPATH=str(tmp_path) + os.pathsep + ROOT)
    files = [os.path.join(HERE, f"test_oracle_{p}.py") for p in pins]
    # run from the planted copy's directory, so that it is the oracle imported
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *files], cwd=str(tmp_path), env=env, capture_output=True, text=True)
    assert r.returncode == 1, f"{name}: no pin failed\n{r.stdout[-2000:]}"
