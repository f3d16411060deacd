"""Mutation check of the oracle's pins.

The oracle is trusted because its CPU tests pin it to facts from outside its
own code: worked examples and traces printed on the pages, closed forms,
exhaustive format tables, invariants.  This file checks that those pins are
strong enough.  Each mutant below plants one plausible mistake in a private
copy of the oracle: a dropped term, a wrong sign or index, an off-by-one, the
wrong rounding, a swapped operand.  The copy's pin tests must then fail.  A
mutant that survives means a hole in the pins.

Every mutant runs in its own scratch directory.  That directory holds copies
of oracle/ and of the oracle's CPU tests.  Nothing in the repository is
modified, and no GPU is involved.  An unmutated copy must pass, which shows
that the harness itself is sound.
"""

import concurrent.futures
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CPP = "oracle/zdp_oracle.cpp"
ACC = "oracle/accounting.py"

# (name, [(file, old text, new text), ...]); each old text occurs exactly once.
MUTANTS = [
    # number formats
    ("bf16 widening shifts by 15",
     [(CPP, "static_cast<uint32_t>(h) << 16", "static_cast<uint32_t>(h) << 15")]),
    ("fp16 subnormal scale 2^-25",
     [(CPP, "static_cast<float>(f), -24);", "static_cast<float>(f), -25);")]),
    ("fp16 exponent bias off by one", [(CPP, "e - 25);", "e - 24);")]),
    ("fp16 infinity read as NaN", [(CPP, "mag = INFINITY;", "mag = NAN;")]),
    ("bf16 rounding truncates",
     [(CPP, "if (rest > 0x8000u || (rest == 0x8000u && (lo & 1u))) lo += 1;", "")]),
    ("bf16 ties away from zero",
     [(CPP, "(rest == 0x8000u && (lo & 1u))", "(rest == 0x8000u)")]),
    ("bf16 NaN becomes infinity", [(CPP, "| 0x7fc0u);", "| 0x7f80u);")]),
    # ownership and the ring order
    ("shard size one too large",
     [(CPP, "int64_t shard_size(int64_t n, int P) { return (n + P - 1) / P; }",
       "int64_t shard_size(int64_t n, int P) { return (n + P) / P; }")]),
    ("owner index shifted by one element",
     [(CPP, "return static_cast<int>(i / S);", "return static_cast<int>((i + 1) / S);")]),
    ("ring sum starts at the owner",
     [(CPP, "float acc = vals[(r + 1) % P];\n  for (int k = 2; k <= P; ++k)",
       "float acc = vals[r % P];\n  for (int k = 1; k < P; ++k)")]),
    ("ring sum drops the owner's gradient",
     [(CPP, "for (int k = 2; k <= P; ++k) acc", "for (int k = 2; k < P; ++k) acc")]),
    ("ring sum runs backwards",
     [(CPP, "acc = acc + vals[(r + k) % P];", "acc = acc + vals[(r + P + 1 - k) % P];")]),
    ("literal ring sends the wrong chunk",
     [(CPP, "int c = ((i - s - shift) % P + P) % P;", "int c = ((i + s - shift) % P + P) % P;")]),
    ("literal all-gather forwards the wrong chunk",
     [(CPP, "int c = ((i + 1 - shift - s) % P + P) % P;", "int c = ((i - shift - s) % P + P) % P;")]),
    ("fused step forgets the averaging scale",
     [(CPP, "g[j] = ring_sum(vals.data(), P, owner_of(i, S)) * scale;",
       "g[j] = ring_sum(vals.data(), P, owner_of(i, S));")]),
    ("reduce-scatter forgets the averaging scale",
     [(CPP, "static_cast<double>(g);\n    shards[i] = g;",
       "static_cast<double>(g);\n    shards[i] = g / scale;")]),
    # AdamW
    ("first bias correction at t+1",
     [(CPP, "a.bc1 = static_cast<float>(1.0 - std::pow(static_cast<double>(b1), static_cast<double>(t)));",
       "a.bc1 = static_cast<float>(1.0 - std::pow(static_cast<double>(b1), static_cast<double>(t + 1)));")]),
    ("second bias correction uses beta1",
     [(CPP, "a.bc2 = static_cast<float>(1.0 - std::pow(static_cast<double>(b2),",
       "a.bc2 = static_cast<float>(1.0 - std::pow(static_cast<double>(b1),")]),
    ("no first bias correction", [(CPP, "const float m_hat = m_new / a.bc1;", "const float m_hat = m_new;")]),
    ("eps inside the square root",
     [(CPP, "std::sqrt(v_hat) + a.eps;", "std::sqrt(v_hat + a.eps);")]),
    ("betas swapped in the first moment",
     [(CPP, "a.b1 * m + a.one_minus_b1 * g;", "a.b2 * m + a.one_minus_b2 * g;")]),
    ("second moment of |g|", [(CPP, "const float g_sq = g * g;", "const float g_sq = std::fabs(g);")]),
    ("update from the old first moment",
     [(CPP, "const float u = m_hat / denom;", "const float u = (m / a.bc1) / denom;")]),
    ("weight decay with the wrong sign",
     [(CPP, "const float w_decayed = w - a.lr_wd * w;", "const float w_decayed = w + a.lr_wd * w;")]),
    ("weight decay on the updated weight",
     [(CPP, "const float w_decayed = w - a.lr_wd * w;\n  w = w_decayed - a.lr * u;",
       "const float w_step = w - a.lr * u;\n  w = w_step - a.lr_wd * w_step;")]),
    ("learning rate missing from the decay",
     [(CPP, "a.lr_wd = lr * wd;", "a.lr_wd = wd;")]),
    # overflow flag, skip and sum of squares
    ("NaN counted as finite",
     [(CPP, "bool is_finite(float x) { return (float_to_bits(x) & 0x7f800000u) != 0x7f800000u; }",
       "bool is_finite(float x) { return std::fabs(x) != INFINITY; }")]),
    ("checked step ignores the flag",
     [(CPP, "if (check_overflow && flag) return 0;", "if (check_overflow && flag && false) return 0;")]),
    ("sum of |g| instead of g^2",
     [(CPP, "ss += static_cast<double>(g[j]) * static_cast<double>(g[j]);",
       "ss += std::fabs(static_cast<double>(g[j]));")]),
    ("sum of squares in fp32",
     [(CPP, "ss += static_cast<double>(g[j]) * static_cast<double>(g[j]);",
       "ss += static_cast<double>(g[j] * g[j]);")]),
    ("sum of squares taken before the scale",
     [(CPP, "ss += static_cast<double>(g[j]) * static_cast<double>(g[j]);",
       "ss += static_cast<double>(g[j] / scale) * static_cast<double>(g[j] / scale);")]),
    ("reduce-scatter sums |g|",
     [(CPP, "ss += static_cast<double>(g) * static_cast<double>(g);\n    shards[i] = g;",
       "ss += std::fabs(static_cast<double>(g));\n    shards[i] = g;")]),
    ("ZeRO++ sum of squares in fp32",
     [(CPP, "ss += static_cast<double>(g) * static_cast<double>(g);\n    const int64_t k = i - base;",
       "ss += static_cast<double>(g * g);\n    const int64_t k = i - base;")]),
    ("ZeRO++ sum of squares skips the owner's rank",
     [(CPP, "vals[q] = dequant_one(gq[q * ld + j], gs[q * sld + i / kQBlock - off / kQBlock]);",
       "vals[q] = q == owner_of(i, S) ? 0.0f : dequant_one(gq[q * ld + j], gs[q * sld + i / kQBlock - off / kQBlock]);")]),
    # the sampled step (the checker of the full-size parity tests)
    ("sampled step ignores the skip", [(CPP, "    if (!skip) {", "    if (true) {")]),
    ("sampled owner from the position in the sample",
     [(CPP, "ring_sum(vals.data(), P, owner_of(idx[j], S)) * scale;",
       "ring_sum(vals.data(), P, owner_of(j, S)) * scale;")]),
    ("sampled step widens every gradient as bf16",
     [(CPP, "for (int q = 0; q < P; ++q) vals[q] = widen(gs[q * k + j], gdt);",
       "for (int q = 0; q < P; ++q) vals[q] = widen(gs[q * k + j], 0);")]),
    # replicas
    ("replicas truncated to bf16",
     [(CPP, "const uint16_t p = float_to_bf16_rne(master[k]);",
       "const uint16_t p = static_cast<uint16_t>(float_to_bits(master[k]) >> 16);")]),
    ("replicas take the pre-update weight",
     [(CPP, "adamw_element(master[k], mk, vk, g[j], a);\n    store_moment(m, k, mdt, mk);\n    store_moment(v, k, mdt, vk);\n    const uint16_t p = float_to_bf16_rne(master[k]);",
       "const float w_old = master[k];\n    adamw_element(master[k], mk, vk, g[j], a);\n    store_moment(m, k, mdt, mk);\n    store_moment(v, k, mdt, vk);\n    const uint16_t p = float_to_bf16_rne(w_old);")]),
    ("only the owner's replica written",
     [(CPP, "for (int q = 0; q < P; ++q) replicas[q * rld + k] = p;",
       "replicas[owner_of(off + j, S) * rld + k] = p;")]),
    # bf16 moments
    ("bf16 moments stored truncated",
     [(CPP, "static_cast<uint16_t*>(base)[k] = float_to_bf16_rne(x);",
       "static_cast<uint16_t*>(base)[k] = static_cast<uint16_t>(float_to_bits(x) >> 16);")]),
    # ZeRO++ block quantization
    ("quantization scale amax/128", [(CPP, "return amax / 127.0f;", "return amax / 128.0f;")]),
    ("quantization truncates", [(CPP, "std::nearbyint(y);", "std::trunc(y);")]),
    ("quantization ties away from zero", [(CPP, "std::nearbyint(y);", "std::round(y);")]),
    ("quantization drops a NaN from the block maximum",
     [(CPP, "if (std::isnan(a)) return std::numeric_limits<float>::quiet_NaN();", "")]),
    ("a NaN quotient clamps to +127", [(CPP, "if (std::isnan(y)) return -127;",
                                        "if (std::isnan(y)) return 127;")]),
    ("quantization clamps at 126", [(CPP, "if (r > 127.0f) r = 127.0f;", "if (r > 126.0f) r = 126.0f;")]),
    ("dequantization reads the next block's scale",
     [(CPP, "x[i] = dequant_one(q[i], scales[i / kQBlock]);",
       "x[i] = dequant_one(q[i], scales[(i + 1) / kQBlock]);")]),
    ("ZeRO++ gradient scale index ignores the range start",
     [(CPP, "gs[q * sld + i / kQBlock - off / kQBlock]", "gs[q * sld + i / kQBlock]")]),
    ("ZeRO++ replicas quantized from the fp32 master",
     [(CPP, "p[j] = bf16_to_float(float_to_bf16_rne(master[k]));", "p[j] = master[k];")]),
    # accounting
    ("fp32 moments counted as 2 bytes", [(ACC, '"m_fp32": 4,', '"m_fp32": 2,')]),
    ("ZeRO-2 shards only the optimizer state",
     [(ACC, "return p + (g + o) / n_gpus", "return p + g + o / n_gpus")]),
    ("ring sends 2p messages", [(ACC, "return 2 * (p - 1) * s", "return 2 * p * s")]),
    ("fused step reads the gradients twice",
     [(ACC, "return P * grad_bytes + state + state + P * param_bytes",
       "return 2 * P * grad_bytes + state + state + P * param_bytes")]),
]

_TEST_FILES = sorted(f for f in os.listdir(os.path.join(ROOT, "tests"))
                     if f.startswith("test_oracle_") and f.endswith(".py")
                     and f != os.path.basename(__file__))


def _copy_tree(dst):
    os.makedirs(os.path.join(dst, "oracle"))
    for f in ("__init__.py", "accounting.py", "zdp_oracle.cpp"):
        shutil.copy(os.path.join(ROOT, "oracle", f), os.path.join(dst, "oracle", f))
    os.makedirs(os.path.join(dst, "tests"))
    for f in ["conftest.py", "harness_cpu.py", *_TEST_FILES]:
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), os.path.join(dst, "tests", "golden"))


def _apply(dst, edits):
    for rel, old, new in edits:
        path = os.path.join(dst, rel)
        text = open(path).read()
        assert text.count(old) == 1, f"{rel}: mutation site must occur once: {old!r}"
        with open(path, "w") as f:
            f.write(text.replace(old, new))


def _run(dst):
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    cmd = [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
           "-m", "not gpu", *[os.path.join("tests", f) for f in _TEST_FILES]]
    r = subprocess.run(cmd, cwd=dst, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, (r.stdout + r.stderr)[-1500:]


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    base = tmp_path_factory.mktemp("mutants")
    jobs = {"unmutated": []}
    jobs.update({name: edits for name, edits in MUTANTS})
    dirs = {}
    for k, (name, edits) in enumerate(jobs.items()):
        d = str(base / f"m{k:02d}")
        _copy_tree(d)
        _apply(d, edits)
        dirs[name] = d
    workers = max(1, min(8, os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as pool:
        futs = {name: pool.submit(_run, d) for name, d in dirs.items()}
        return {name: f.result() for name, f in futs.items()}


def test_unmutated_copy_passes(outcomes):
    rc, tail = outcomes["unmutated"]
    assert rc == 0, tail


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_mutant_is_caught(outcomes, name):
    rc, tail = outcomes[name]
    # exit code 1: tests ran and at least one failed (not a build or collection error)
    assert rc == 1, f"mutant survived or broke the harness (exit {rc}):\n{tail}"
