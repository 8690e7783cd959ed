"""The oracle's pins have teeth: each plausible mistake below is planted, one at a time,
in a scratch copy of the oracle source; the copy is rebuilt and the pin suite
(tests/test_oracle_pins.py) must fail on it. Everything runs on the CPU in a temporary
directory; the repository's oracle is never modified."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "zpp_oracle.c")

# (name, original text, planted mistake)
MUTANTS = [
    ("qmax off by one", "const float qmax = (float)((1 << (bits - 1)) - 1);",
     "const float qmax = (float)((1 << (bits - 1)));"),
    ("round half away from zero", "double t = nearbyint((double)v[i] * (double)inv);",
     "double t = round((double)v[i] * (double)inv);"),
    ("product rounded to fp32 first", "double t = nearbyint((double)v[i] * (double)inv);",
     "double t = nearbyint((double)(v[i] * inv));"),
    ("divide instead of multiply", "double t = nearbyint((double)v[i] * (double)inv);",
     "double t = nearbyint((double)(v[i] / scale));"),
    ("nibbles swapped", "out[i] = (uint8_t)(lo | (hi << 4));", "out[i] = (uint8_t)(hi | (lo << 4));"),
    ("INT4 not sign-extended", "return nib >= 8 ? nib - 16 : nib;", "return nib;"),
    ("zero rule ignores overflowing inverse", "if (amax == 0.0f || !isfinite(inv)) {",
     "if (amax == 0.0f) {"),
    ("tail block treated as full", "int64_t lo = b * block, len = (n - lo < block) ? n - lo : block;",
     "int64_t lo = b * block, len = block;"),
    ("dequant uses the wrong block scale",
     "float v = (float)code_at(codes, bits, i) * scales[i / block];",
     "float v = (float)code_at(codes, bits, i) * scales[(i + 1) / block];"),
    ("no slice reorder", "return l_d * N + n_d;", "return n_d * M + l_d;"),
    ("hop 1 reads the wrong chunk", "int64_t idx = (int64_t)l * C + e; /* chunk l",
     "int64_t idx = (int64_t)lp * C + e; /* chunk l"),
    ("hop 2 reads the wrong slice", "int64_t idx = (int64_t)n * S + e; /* slice n",
     "int64_t idx = (int64_t)np * S + e; /* slice n"),
    ("hop 2 transposed source", "static int64_t hop2_source(int np, int M, int l) { return (int64_t)np * M + l; }",
     "static int64_t hop2_source(int np, int M, int l) { return (int64_t)l * M + np; }"),
    ("hop 1 drops a source", "for (int lp = 0; lp < M; ++lp) {", "for (int lp = 1; lp < M; ++lp) {"),
    ("hop 1 subtracts", "scales[src * (E / block) + idx / block], a);",
     "-scales[src * (E / block) + idx / block], a);"),
    ("hop sums rounded twice",
     "a = fmaf((float)code_at(codes + src * or_code_bytes(E, bits), bits, idx),\n"
     "                   scales[src * (E / block) + idx / block], a);",
     "a = a + (float)code_at(codes + src * or_code_bytes(E, bits), bits, idx) *\n"
     "                   scales[src * (E / block) + idx / block];"),
    ("average not applied", "store_value(out, out_dtype, i, sum[i] * post_scale);",
     "store_value(out, out_dtype, i, sum[i]);"),
    ("fp16 truncates", "double m = nearbyint(a * ldexp(1.0, 10 - E));",
     "double m = floor(a * ldexp(1.0, 10 - E));"),
    ("bf16 rounds ties up", "if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u))) hi += 1u;",
     "if (lo >= 0x8000u) hi += 1u;"),
]


def _copy_repo(dst):
    def ignore(path, names):
        return {n for n in names if n in (".git", "__pycache__", "_build",
                                          ".pytest_cache") or n.endswith((".so", ".o"))}
    for d in ("oracle", "tests", "quantized_zero_communication_gb300"):
        shutil.copytree(os.path.join(ROOT, d), os.path.join(dst, d), ignore=ignore)
    shutil.copy(os.path.join(ROOT, "include", "zpp.h"), dst)


@pytest.mark.parametrize("name,orig,bad", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(name, orig, bad, tmp_path):
    src = open(SRC).read()
    assert src.count(orig) >= 1, f"mutation site not found: {name}"
    _copy_repo(str(tmp_path))
    with open(tmp_path / "oracle" / "zpp_oracle.c", "w") as f:
        f.write(src.replace(orig, bad, 1))
    # the planted source must still compile: a mutant is caught by a pin, not by the compiler
    from oracle import build as obuild
    cc = subprocess.run(["gcc", *obuild.BASE_FLAGS, str(tmp_path / "oracle" / "zpp_oracle.c"),
                         "-o", str(tmp_path / "probe.so"), "-lm"], capture_output=True, text=True)
    assert cc.returncode == 0, cc.stderr
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, capture_output=True, text=True,
                       timeout=600)
    # 1: a pin failed; negative: the planted mistake crashed the oracle (e.g. an overrun)
    assert r.returncode == 1 or r.returncode < 0, f"pins did not catch: {name}\n{r.stdout[-500:]}"
