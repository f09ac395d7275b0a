"""Mutation check of the oracle's pins: plant one plausible mistake at a time
in a copy of oracle/ar_oracle.c and confirm that the CPU pin tests
(tests/test_oracle_*.py) fail on it.

Run by hand (not collected by pytest):  python tests/oracle_mutations.py
It first runs the pins on an unmodified copy (which must pass), then once per
mistake below, and prints CAUGHT or MISSED for each; the exit status is 0 only
if every mistake is caught.  The copies live under oracle/_build/ and are
removed afterwards.
"""

import pathlib
import shutil
import subprocess
import sys
import tempfile

ROOT = pathlib.Path(__file__).resolve().parents[1]

# (name, function the mistake is planted in, text there, replacement, occurrences to replace)
MUTATIONS = [
    ("bf16 rounding: ties away from zero", "orc_f32_to_bf16",
     "if (drop > 0x8000u || (drop == 0x8000u && (keep & 1u)))", "if (drop >= 0x8000u)", 1),
    ("fp16 rounding: ties away from zero", "orc_f32_to_f16",
     "if (rem > half || (rem == half && (r & 1u)))", "if (rem >= half)", 1),
    ("fp16 subnormal quantum off by one binade", "orc_f32_to_f16",
     "int q = (E >= -14) ? E - 10 : -24;", "int q = (E >= -14) ? E - 10 : -25;", 1),
    ("fp16 sign lost", "orc_f32_to_f16", "return (uint16_t)(sign | bits);", "return (uint16_t)(bits);", 1),
    ("sum starts at rank 0's value instead of +0", "orc_all_reduce",
     "float acc = 0.0f;\n        for (int r = 0; r < n; ++r)",
     "float acc = widen(in[0], i, dt);\n        for (int r = 1; r < n; ++r)", 1),
    ("last rank dropped from the sum", "orc_all_reduce",
     "for (int r = 0; r < n; ++r)\n            acc = acc + widen(in[r], i, dt);",
     "for (int r = 0; r < n - 1; ++r)\n            acc = acc + widen(in[r], i, dt);", 1),
    ("chunk not rounded up to a 16-byte vector", "orc_chunk_elems",
     "return (per + q - 1) / q * q;", "return per + 0 * q;", 1),
    ("reduce-scatter sums the wrong chunk", "orc_reduce_scatter",
     "chunk_range(r, C, N, &lo, &hi);", "chunk_range((r + 1) % n, C, N, &lo, &hi);", 1),
    ("ring rotation reversed", "orc_ring", "((r - s) % n + n) % n", "((r + s) % n + n) % n", 2),
    ("ring rounds the wrong completed chunk", "orc_ring",
     "chunk_range((r + 1) % n, C, N, &lo, &hi);\n        for (size_t i = lo; i < hi; ++i)\n            narrow(",
     "chunk_range(r % n, C, N, &lo, &hi);\n        for (size_t i = lo; i < hi; ++i)\n            narrow(", 1),
    ("ring all-gather passes the wrong chunk", "orc_all_gather_ring",
     "((r + 1 - s) % n + n) % n", "((r - s) % n + n) % n", 2),
    ("LL unpack ignores the flag", "orc_ll_unpack",
     "if (get_u32(lines + 8 * i + 4) != step) { ++bad; continue; }", "if (0) { ++bad; continue; }", 1),
    ("LL128 flag at the wrong offset", "orc_ll128_pack", "put_u64(line + 120, step);",
     "put_u64(line + 112, step);", 1),
    ("LL reduce consumes a line whatever its flags", "orc_ll_reduce",
     "ok = ok && get_u32(in[r] + 8 * i + 4) == step;", "ok = ok || 1;", 1),
    ("hop-rounded ring rotation reversed", "orc_ring_rounded", "((r - s) % n + n) % n", "((r + s) % n + n) % n", 2),
    ("hop-rounded ring one hop short", "orc_ring_rounded",
     "for (int s = 0; s < n - 1; ++s) {", "for (int s = 0; s < n - 2; ++s) {", 1),
    ("hop-rounded ring gathers the wrong chunk", "orc_ring_rounded",
     "chunk_range((r + 1) % n, C, N, &lo, &hi);\n        if (hi > lo)",
     "chunk_range(r % n, C, N, &lo, &hi);\n        if (hi > lo)", 1),
    ("tree pairs cyclically instead of by XOR", "orc_tree", "int p = r ^ d;", "int p = (r + d) % n;", 1),
    ("tree skips level 0", "orc_tree", "for (int d = 1; d < n; d <<= 1) {", "for (int d = 2; d < n; d <<= 1) {", 1),
    ("tree adds a rank to itself", "orc_tree", "widen(cur, (size_t)p * N + i, dt);",
     "widen(cur, (size_t)r * N + i, dt);", 1),
]


def _function_span(src: str, name: str) -> tuple[int, int]:
    """[start, end) of the definition of `name` in the C source: from its
    signature to the next top-level closing brace."""
    marks = [i for i in range(len(src)) if src.startswith(name + "(", i) and (i == 0 or not src[i - 1].isalnum())]
    for start in marks:
        line_start = src.rfind("\n", 0, start) + 1
        if src[line_start:start].strip() and not src[line_start:start].lstrip().startswith("/*"):
            brace = src.find("\n{", start)
            end = src.find("\n}", brace)
            if brace != -1 and end != -1 and src.find(";", start, brace) == -1:
                return line_start, end + 2
    raise KeyError(name)


def _run_pins(tmp: pathlib.Path) -> tuple[bool, str]:
    # the oracle's pin tests (this check's own test file is named apart from them)
    tests = sorted(str(p.relative_to(tmp)) for p in (tmp / "tests").glob("test_oracle_*.py"))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider", *tests],
                       cwd=tmp, capture_output=True, text=True)
    out = r.stdout.strip().splitlines()
    return r.returncode == 0, (out[-1] if out else r.stderr.strip()[-200:])


def _copy(base: pathlib.Path) -> pathlib.Path:
    tmp = pathlib.Path(tempfile.mkdtemp(prefix="mutant_", dir=base))
    for d in ("oracle", "workloads", "tests"):
        shutil.copytree(ROOT / d, tmp / d, ignore=shutil.ignore_patterns("_build", "__pycache__"))
    return tmp


def main() -> int:
    base = ROOT / "oracle" / "_build"
    base.mkdir(exist_ok=True)
    tmp = _copy(base)
    try:
        ok, last = _run_pins(tmp)
    finally:
        shutil.rmtree(tmp)
    print(f"{'PASS  ' if ok else 'FAIL  '} unmodified oracle: {last}")
    if not ok:
        return 2
    missed = 0
    for name, fn, old, new, count in MUTATIONS:
        tmp = _copy(base)
        try:
            src_path = tmp / "oracle" / "ar_oracle.c"
            src = src_path.read_text()
            a, b = _function_span(src, fn)
            body = src[a:b]
            if body.count(old) < count:
                raise RuntimeError(f"{name}: text not found in {fn}")
            src_path.write_text(src[:a] + body.replace(old, new, count) + src[b:])
            ok, last = _run_pins(tmp)
        finally:
            shutil.rmtree(tmp)
        missed += ok
        print(f"{'MISSED' if ok else 'CAUGHT'}  {name}: {last}")
    print(f"{len(MUTATIONS) - missed} of {len(MUTATIONS)} planted mistakes caught")
    return 1 if missed else 0


if __name__ == "__main__":
    sys.exit(main())
