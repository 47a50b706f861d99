"""The oracle's pins must catch plausible mistakes: each case plants one bug
in a copy of oracle/lora_oracle.c (a dropped term, a wrong index or sign, an
off-by-one, a broken rule), builds it, and runs tests/test_oracle_pins.py
against it; the pins must fail.  CPU only; nothing here touches the GPU path."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "lora_oracle.c")

# (name, exact text in lora_oracle.c, replacement)
MUTATIONS = [
    ("map_tokens_accepts_L", "if (l >= 0 && l < L) {", "if (l >= 0 && l <= L) {"),
    ("map_tokens_no_bad_count", "if (l != -1) bad++;", "if (0) bad++;"),
    ("segments_no_overlap_rule", "int overlaps = s0 < prev_end;", "int overlaps = 0;"),
    ("segments_no_range_rule", "if (s0 < 0 || n < 0 || s0 + n > T) { *err |= 1; continue; }",
     "if (s0 < 0 || n < 0) { *err |= 1; continue; }"),
    ("segments_bad_id_kept", "if (!(l >= -1 && l < L)) { bad++; l = -1; }",
     "if (!(l >= -1 && l < L)) { bad++; }"),
    ("group_unstable_order",
     "for (int32_t t = 0; t < T; ++t)\n                if (lora_of[t] == l) perm[pos++] = t;",
     "for (int32_t t = T - 1; t >= 0; --t)\n                if (lora_of[t] == l) perm[pos++] = t;"),
    ("group_full_tiles_only",
     "int32_t n = group_count[i] - p < tile ? group_count[i] - p : tile;", "int32_t n = tile;"),
    ("group_inactive_first_tile_lora", "tiles[4 * k + 0] = -1;", "tiles[4 * k + 0] = 0;"),
    ("shrink_drops_scale", "v = scale * acc;", "v = acc;"),
    ("shrink_transposed_rows", "const double *a = A + ((int64_t)l * S * R + j) * H;",
     "const double *a = A + ((int64_t)l * S * R + (int64_t)i * S + s) * H;"),
    ("shrink_rank_off_by_one", "if (l >= 0 && i < r) {", "if (l >= 0 && i <= r && i < R) {"),
    ("shrink_ignores_add", "*yy = (add ? *yy : 0.0) + v;", "*yy = v;"),
    ("shrink_wrong_adapter", "const double *a = A + ((int64_t)l * S * R + j) * H;",
     "const double *a = A + ((int64_t)(l > 0 ? l - 1 : 0) * S * R + j) * H;"),
    ("shrink_sign", "acc += xr[h] * a[h];", "acc -= xr[h] * a[h];"),
    ("expand_transposed_B", "acc += yr[i] * b[i];",
     "acc += yr[i] * B[s][((int64_t)l * R + i) * N[s] + n];"),
    ("expand_ignores_offset", "double *o = out + (int64_t)t * ldo + off[s] + n;",
     "double *o = out + (int64_t)t * ldo + n;"),
    ("expand_zeroes_inactive_with_add", "if (!add) *o = 0.0;", "*o = 0.0;"),
    ("expand_reads_slice0_y", "(int64_t)t * ldy + (int64_t)s * y_stride;", "(int64_t)t * ldy;"),
    ("expand_drops_scale", "*o = (add ? *o : 0.0) + scale * acc;", "*o = (add ? *o : 0.0) + acc;"),
    ("expand_ignores_rank", "for (int32_t i = 0; i < r; ++i) acc += yr[i] * b[i];",
     "for (int32_t i = 0; i < R; ++i) acc += yr[i] * b[i];"),
    ("rank_no_lower_clamp", "if (r < 0) r = 0;", "if (r < 0) r = -r;"),
]


def _build(src_text, tmp_path):
    c = tmp_path / "mutant.c"
    so = tmp_path / "libmutant.so"
    c.write_text(src_text)
    subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
                    "-ffp-contract=off", str(c), "-o", str(so)], check=True)
    return str(so)


def _run_pins(lib):
    env = dict(os.environ, LORA_ORACLE_LIB=lib, OMP_NUM_THREADS="2")
    return subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests",
                                                                          "test_oracle_pins.py"),
                           "-x", "-q", "-p", "no:cacheprovider"],
                          cwd=ROOT, env=env, capture_output=True, text=True)


def test_unmutated_copy_passes(tmp_path):
    """Control: the pins pass on an unmodified copy built the same way."""
    r = _run_pins(_build(open(SRC).read(), tmp_path))
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_mutation(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: mutation site not found exactly once"
    r = _run_pins(_build(src.replace(old, new), tmp_path))
    assert r.returncode != 0, f"mutation {name} survived the oracle pins"
