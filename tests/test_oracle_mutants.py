"""The pins bite: each case plants one plausible mistake in a copy of the oracle's C
source (a dropped term, a wrong sign, index or bound, swapped operands, a wrong
format constant), builds that copy, and runs the pins against it; at least one pin
must fail (a test failure, not a crash).  Every planted change keeps the oracle's
memory accesses inside its buffers."""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "paged_ref.c")

# (name, text in the source, replacement, occurrence to change: 0 = the first)
MUTANTS = [
    # decode attention
    ("decode: score scale dropped", "\n        z[j] = scale * acc;", "\n        z[j] = acc;", 0),
    ("decode: max shift of the wrong sign", "\n        z[j] = exp(z[j] - zmax);", "\n        z[j] = exp(z[j] + zmax);", 0),
    ("decode: softmax not normalised", "for (int64_t j = 0; j < L; ++j) z[j] /= den;", ";", 0),
    ("decode: query heads interleaved over KV heads",
     "\n    for (int64_t h = k * group; h < (k + 1) * group; ++h) {",
     "\n    for (int64_t h = k; h < num_heads; h += num_kv_heads) {", 0),
    ("decode: keys read from the value cache", "orc_load(key_cache, base + d, kv_dtype) * ks;",
     "orc_load(value_cache, base + d, kv_dtype) * ks;", 0),
    ("decode: values read from the key cache", "orc_load(value_cache, base + d, kv_dtype) * vs;",
     "orc_load(key_cache, base + d, kv_dtype) * vs;", 0),
    ("decode: offset inside the block off by one", "(j % block_size) * cs_token", "((j + 1) % block_size) * cs_token", 0),
    ("decode: newest position not attended", "int64_t L = Lctx - j0;", "int64_t L = Lctx - j0 - 1;", 0),
    ("decode: block-table row stride dropped", "block_tables[s * max_blocks_per_seq + j / block_size]",
     "block_tables[s + j / block_size]", 0),
    ("decode: window one position too wide", "Lctx - sliding_window : 0", "Lctx - sliding_window - 1 : 0", 0),
    ("decode: per-head key scale ignored", "k_head_scales ? (double)k_head_scales[k] : k_scale", "k_scale", 0),
    # number formats
    ("e4m3: exponent bias 8", "ldexp(1.0 + m / 8.0, e - 7)", "ldexp(1.0 + m / 8.0, e - 8)", 0),
    ("e4m3: subnormal step 2^-10", "ldexp((double)m, -9)", "ldexp((double)m, -10)", 0),
    ("e4m3: ties to the odd code", "((lo + 1) & 1) == 0", "((lo + 1) & 1) == 1", 0),
    ("e4m3: overflow to NaN, not saturated", "return (uint8_t)(sign | 0x7E);", "return (uint8_t)(sign | 0x7F);", 0),
    ("bf16: bits shifted by 15", "(uint32_t)bits << 16", "(uint32_t)bits << 15", 0),
    # cache write
    ("write: slot offset off by one", "off = slot % block_size;", "off = (slot + 1) % block_size;", 0),
    ("write: scale multiplies", "float yk = xk / ksh;", "float yk = xk * ksh;", 0),
    ("write: amax of signed values", "double ak = fabs(orc_load(key, src + d, src_dtype))",
     "double ak = (orc_load(key, src + d, src_dtype))", 0),
    # copy-on-write
    ("copy: source and destination swapped",
     "memmove((char*)cache + dst * block_bytes, (const char*)cache + src * block_bytes,",
     "memmove((char*)cache + src * block_bytes, (const char*)cache + dst * block_bytes,", 0),
    # prefill
    ("prefill: query sees one position less", "int64_t pos = L - n + i;", "int64_t pos = L - n + i - 1;", 0),
    ("prefill: every row uses the last query", "const int64_t qoff = ((q0 + i) * num_heads + h) * head_dim;",
     "const int64_t qoff = ((q0 + n - 1) * num_heads + h) * head_dim;", 0),
    ("prefill: score scale dropped", "\n          z[j] = scale * acc;", "\n          z[j] = acc;", 0),
    ("prefill: no causal mask", "int64_t pos = L - n + i;", "int64_t pos = L - 1;", 0),
    ("prefill: keys scaled by the value scale", "orc_load(key_cache, base + d, kv_dtype) * k_scale;",
     "orc_load(key_cache, base + d, kv_dtype) * v_scale;", 0),
    # more decode, format and write mistakes
    ("prefill: query heads interleaved over KV heads",
     "for (int64_t h = k * group; h < (k + 1) * group; ++h) {",
     "for (int64_t h = k; h < num_heads; h += num_kv_heads) {", 1),
    ("prefill: max shift of the wrong sign", "z[j] = exp(z[j] - zmax);", "z[j] = exp(z[j] + zmax);", 1),
    ("prefill: softmax not normalised", "for (int64_t j = 0; j <= pos; ++j) z[j] /= den;", ";", 0),
    ("prefill: values read from the key cache",
     "V[j * head_dim + d] = orc_load(value_cache, base + d, kv_dtype) * v_scale;",
     "V[j * head_dim + d] = orc_load(key_cache, base + d, kv_dtype) * v_scale;", 0),
    ("prefill: offset inside the block off by one", "(j % block_size) * cs_token",
     "((j + 1) % block_size) * cs_token", 1),
    ("prefill: block-table row stride dropped", "block_tables[s * max_blocks_per_seq + j / block_size]",
     "block_tables[s + j / block_size]", 1),
    ("prefill: own position left out of the weighted sum",
     "for (int64_t j = 0; j <= pos; ++j)\n          for (int64_t d = 0; d < head_dim; ++d) o[d] += z[j]",
     "for (int64_t j = 0; j < pos; ++j)\n          for (int64_t d = 0; d < head_dim; ++d) o[d] += z[j]", 0),
    ("decode: keys scaled by the value scale", "orc_load(key_cache, base + d, kv_dtype) * ks;",
     "orc_load(key_cache, base + d, kv_dtype) * vs;", 0),
    ("decode: every KV head takes head 0's scale", "k_head_scales ? (double)k_head_scales[k]",
     "k_head_scales ? (double)k_head_scales[0]", 0),
    ("decode: window start ignored", "(sliding_window > 0 && Lctx > sliding_window) ? Lctx - sliding_window : 0",
     "0", 0),
    ("e4m3: sign dropped on decode", "return sign ? -mag : mag;", "return mag;", 0),
    ("e4m3: NaN encoded as zero", "if (isnan(y)) return 0x7F;", "if (isnan(y)) return 0x00;", 0),
    ("bf16: bits taken as the low half", "(uint32_t)bits << 16", "(uint32_t)bits", 0),
    ("write: value codes stored in the key cache",
     "((uint8_t*)value_cache)[dst + d] = orc_f32_to_e4m3(yv);", "((uint8_t*)key_cache)[dst + d] = orc_f32_to_e4m3(yv);", 0),
    ("write: amax forgets a NaN", "if (k_amax && (isnan(ak) || ak > k_amax[h])) k_amax[h] = ak;",
     "if (k_amax && (ak > k_amax[h])) k_amax[h] = ak;", 0),
    ("copy: half of each block", "(size_t)block_bytes);", "(size_t)block_bytes / 2);", 0),
    ("decode: every head uses its group's first query", "const int64_t qoff = (s * num_heads + h) * head_dim;",
     "const int64_t qoff = (s * num_heads + k * group) * head_dim;", 0),
    ("decode: every sequence reads sequence 0's table", "block_tables[s * max_blocks_per_seq + j / block_size]",
     "block_tables[0 * max_blocks_per_seq + j / block_size]", 0),
    ("e4m3: encoder truncates", "lo = lo + 1;", ";", 0),
    ("write: value amax read from the keys", "av = fabs(orc_load(value, src + d, src_dtype))",
     "av = fabs(orc_load(key, src + d, src_dtype))", 0),
]


def _plant(text, old, new, which):
    start = -1
    for _ in range(which + 1):
        start = text.find(old, start + 1)
        assert start >= 0, f"{old!r} not found"
    return text[:start] + new + text[start + len(old):]


def _run_pins(tmp_path, i, name, old, new, which):
    d = tmp_path / f"m{i}"
    d.mkdir()
    with open(SRC) as f:
        text = f.read()
    src = d / "paged_ref.c"
    src.write_text(_plant(text, old, new, which))
    env = dict(os.environ, PKV_ORACLE_MUTANT_SRC=str(src), PKV_ORACLE_MUTANT_BUILD=str(d / "build"),
               OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q", "-m", "not gpu",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode, r.stdout[-1500:] + r.stderr[-500:]


def test_mutant_table_plants_distinct_changes():
    with open(SRC) as f:
        text = f.read()
    seen = set()
    for name, old, new, which in MUTANTS:
        changed = _plant(text, old, new, which)
        assert changed != text and changed not in seen, name
        seen.add(changed)


def test_every_planted_mistake_fails_a_pin(tmp_path):
    """Plus a control: an unchanged copy, built and loaded the same way, passes every pin."""
    control = ("control: unchanged copy", "int orc_max_threads(void) {", "int orc_max_threads(void) {", 0)
    cases = [(i, *m) for i, m in enumerate(MUTANTS + [control])]
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda a: _run_pins(tmp_path, *a), cases))
    *mutants, (_, rc_control, out_control) = results
    assert rc_control == 0, out_control
    survivors = [name for name, rc, _ in mutants if rc == 0]
    crashed = [(name, rc, out) for name, rc, out in mutants if rc != 0 and (rc != 1 or " failed" not in out)]
    assert not survivors, f"no pin fails for: {survivors}"
    assert not crashed, f"crashed or did not build instead of failing a pin: {crashed}"
