"""Mutation check of the oracle's pins (CPU only).

Each case copies ``oracle/zp_oracle.c``, plants ONE plausible mistake (a
dropped term, a wrong sign or index, a transposed operand), compiles the copy
into a temporary library and runs every pin against it.  At least one pin must
fail; a mutant that survives means the pins leave that part of the oracle
unchecked.  The real oracle is never modified.
"""
import os
import subprocess
import tempfile

import pytest

import oracle
from tests import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "zp_oracle.c")

MUTANTS = [
    ("causal mask dropped", "int visible = C + i + 1;", "int visible = T;"),
    ("wrong logit scale", "double scale = 1.0 / sqrt((double)d);\n    double *logit",
     "double scale = 1.0 / (double)d;\n    double *logit"),
    ("averaged over w only", "imp[j] /= (double)(w * G);", "imp[j] /= (double)w;"),
    ("query rows transposed", "Q + (size_t)(g * w + i) * d", "Q + (size_t)(i * G + g) * d"),
    ("softmax sum over candidates only",
     "for (int j = 0; j < visible; ++j)\n                S += exp(logit[j] - m);",
     "for (int j = 0; j < C; ++j)\n                S += exp(logit[j] - m);"),
    ("redundancy divided by b", "red[base + j] = f > 1 ? sum / (double)(f - 1) : 0.0;",
     "red[base + j] = f > 1 ? sum / (double)f : 0.0;"),
    ("partial block divided by b-1", "red[base + j] = f > 1 ? sum / (double)(f - 1) : 0.0;",
     "red[base + j] = f > 1 ? sum / (double)(b - 1) : 0.0;"),
    ("prefill: excess blocks kept", "int32_t dst = p < N ? dst_table[(size_t)r * N + p] : -1;",
     "int32_t dst = p < N ? dst_table[(size_t)r * N + p] : src;"),
    ("prefill: length rounded up to whole blocks",
     "int T = J->unit_len ? J->unit_len[row] : N * b;",
     "int T = J->unit_len ? (J->unit_len[row] + b - 1) / b * b : N * b;"),
    ("prefill: short request accepted", "if (T < N * b || T > stride * b)",
     "if (T > stride * b)"),
    ("prefill: released blocks pushed before the pops", "int next_free = free_count - n_pops;",
     "int next_free = free_count;"),
    ("prefill: shared block rewritten in place", "if (refcount[src] > 1) {\n                if (taken",
     "if (refcount[src] > 2) {\n                if (taken"),
    ("self included in redundancy", "if (k == j)\n                    continue;", ""),
    ("squared norm", "norm[j] = sqrt(dot_bf16(kj, kj, d));", "norm[j] = dot_bf16(kj, kj, d);"),
    ("zero-norm guard one-sided", "if (norm[j] > 0.0 && norm[k] > 0.0)", "if (norm[j] > 0.0)"),
    ("lambda sign flipped", "score[j] = imp[j] - lambda * red[j];",
     "score[j] = imp[j] + lambda * red[j];"),
    ("tie-break reversed", "return a < b;", "return a > b;"),
    ("window shifted", "kept[o++] = C + i;", "kept[o++] = C + i - 1;"),
    ("shared block rewritten in place", "if (refcount[blk] > 1) {", "if (refcount[blk] > 2) {"),
    ("pop from the bottom of the stack", "int32_t t = free_ids[free_count - 1 - pops];",
     "int32_t t = free_ids[pops];"),
    ("freed block not pushed", "free_ids[top++] = src;", "(void)src;"),
    ("freed block pushed before the pops", "int top = free_count - n_pops;",
     "int top = free_count;"),
    ("compaction copies identity rows",
     "memcpy(J->kout[l] + off, K + (size_t)kept[j] * d", "memcpy(J->kout[l] + off, K + (size_t)j * d"),
    ("V compaction copies K", "memcpy(J->vout[l] + off, V + (size_t)kept[j] * d",
     "memcpy(J->vout[l] + off, K + (size_t)kept[j] * d"),
    ("decode without scale", "logit[t] = scale * dot_bf16(qv, k, d);",
     "logit[t] = dot_bf16(qv, k, d);"),
    ("decode wrong kv head", "int h = hq / G;", "int h = hq % Hkv;"),
    ("bf16 rounding truncates", "double q = rint(ax / spacing);",
     "double q = floor(ax / spacing);"),
    ("append: shared tail written in place", "if (blk < 0 || refcount[blk] > 1) {\n            int32_t fresh",
     "if (blk < 0) {\n            int32_t fresh"),
    ("append: copy-on-write one row short",
     "memcpy(kpool[l] + to, kpool[l] + from, sizeof(uint16_t) * (size_t)slot * d);",
     "memcpy(kpool[l] + to, kpool[l] + from, sizeof(uint16_t) * (size_t)(slot > 0 ? slot - 1 : 0) * d);"),
    ("append: V not copied on write",
     "memcpy(vpool[l] + to, vpool[l] + from, sizeof(uint16_t) * (size_t)slot * d);", ""),
    ("append: original keeps its reference",
     "                refcount[blk] -= 1;\n            }\n            refcount[fresh] = 1;",
     "            }\n            refcount[fresh] = 1;"),
    ("append: pop from the bottom", "int32_t fresh = free_ids[--fc];",
     "int32_t fresh = free_ids[*free_count - fc--];"),
    ("append: trigger one token early", "if (n_max > 0 && p + 1 == n_max * b) {",
     "if (n_max > 0 && p + 2 == n_max * b) {"),
    ("append: length not advanced", "lengths[row] = p + 1;", "lengths[row] = p;"),
    ("append: full row accepted", "if (p < 0 || p >= stride * b || (n_max > 0 && p >= n_max * b))",
     "if (p < 0 || p >= stride * b)"),
    ("append: new row in the next slot",
     "size_t to = (((size_t)blk * Hkv + h) * b + p % b) * d;",
     "size_t to = (((size_t)blk * Hkv + h) * b + (p + 1) % b) * d;"),
    ("global redundancy over T", "red[j] = T > 1 ? sum / (double)(T - 1) : 0.0;",
     "red[j] = T > 1 ? sum / (double)T : 0.0;"),
    ("global redundancy includes self",
     "if (k == j || norm[j] == 0.0 || norm[k] == 0.0)\n                continue;",
     "if (norm[j] == 0.0 || norm[k] == 0.0)\n                continue;"),
    ("alloc pops from the bottom", "int32_t t = free_ids[--fc];",
     "int32_t t = free_ids[*free_count - fc--];"),
    ("release pushes every reference", "if (--refcount[*entry] == 0)\n                free_ids[fc++] = *entry;",
     "--refcount[*entry];\n                free_ids[fc++] = *entry;"),
    ("release keeps the entries", "            *entry = -1;\n        }\n        lengths[row] = 0;",
     "        }\n        lengths[row] = 0;"),
    ("fork without a reference", "            if (blk >= 0)\n                refcount[blk] += 1;", ""),
    ("length check dropped", "if (lengths[row] != N * b)\n            return ZPO_ERR_INVALID_ARG;",
     ""),
]


def _mutant_lib(tmpdir, old, new):
    with open(SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    path = os.path.join(tmpdir, "mut.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    out = os.path.join(tmpdir, "libmut.so")
    subprocess.run(["gcc", *oracle.GCC_FLAGS, "-w", "-o", out, path, "-lm", "-lpthread"],
                   check=True)
    return out


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new):
    with tempfile.TemporaryDirectory() as tmp:
        orc = oracle.load(_mutant_lib(tmp, old, new))
        caught = []
        for pin in oracle_pins.ALL_PINS:
            try:
                pin(orc)
            except (AssertionError, FloatingPointError, ValueError, IndexError) as e:
                caught.append(pin.__name__)
        assert caught, f"mutant '{name}' passes every pin"
