"""Planted mistakes: each mutant is a copy of oracle.c with one plausible error
(a dropped term, a wrong sign or index, a transposed operand).  The pins in
test_oracle_pins.py must reject every one of them.  CPU only; the mutants are
built in a temporary directory and never touch the real oracle build."""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import oracle
from tests import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, exact text in oracle.c, replacement)
MUTANTS = [
    ("gqa_head_mapping", "h / G, key_cache, value_cache, Hk, D, S, NB, scale,\n                          dtype) != 0;\n    }\n    return bad;\n}\n\n/* ---- FP8 (E4M3) KV cache",
     "h % Hk, key_cache, value_cache, Hk, D, S, NB, scale,\n                          dtype) != 0;\n    }\n    return bad;\n}\n\n/* ---- FP8 (E4M3) KV cache"),
    ("scale_dropped", "s[t] = scale * dot;", "s[t] = dot;"),
    ("softmax_sign", "double w = exp(s[t] - m);", "double w = exp(m - s[t]);"),
    ("causal_off_by_one", "P + j + 1, bt_row", "P + j, bt_row"),
    ("slot_offset_swapped", "int64_t blk = slot / S, off = slot % S;\n        for (int h = 0; h < Hk; ++h) {\n            for (int d",
     "int64_t blk = slot % S, off = slot / S;\n        for (int h = 0; h < Hk; ++h) {\n            for (int d"),
    ("fp8_slot_offset_swapped", "int64_t blk = slot / S, off = slot % S;\n        for (int h = 0; h < Hk; ++h) {\n            float kinv",
     "int64_t blk = slot % S, off = slot / S;\n        for (int h = 0; h < Hk; ++h) {\n            float kinv"),
    ("page_offset_wrong", "const uint16_t* k = kc + cache_index(blk, kvh, t % S, Hk, S, D);",
     "const uint16_t* k = kc + cache_index(blk, kvh, t / S, Hk, S, D);"),
    ("value_from_key_pool", "const uint16_t* v = vc + cache_index(",
     "const uint16_t* v = kc + cache_index("),
    ("merge_sign", "double c = exp(mp[p] - M);", "double c = exp(M - mp[p]);"),
    ("f16_exponent_bias", "ldexp((double)(1024 + f), e - 25)", "ldexp((double)(1024 + f), e - 24)"),
    ("bf16_mantissa_bits", "int f = b & 0x7f;", "int f = b & 0x3f;"),
    ("copy_src_dst_swapped",
     "key_caches[l][dst * block_elems + e] = key_caches[l][src * block_elems + e];",
     "key_caches[l][src * block_elems + e] = key_caches[l][dst * block_elems + e];"),
    ("prefill_prior_len", "int64_t P = context_lens[i] - C;", "int64_t P = context_lens[i] - C + 1;"),
    ("pack_layer_kv_swapped", "uint16_t* st = staging + (((int64_t)l * 2 + kv) * nblk + i) * slab;",
     "uint16_t* st = staging + (((int64_t)kv * L + l) * nblk + i) * slab;"),
    ("unpack_direction", "if (unpack) pool[(int64_t)b * slab + e] = st[e];",
     "if (!unpack) pool[(int64_t)b * slab + e] = st[e];"),
    ("e4m3_exponent_bias", "ldexp((double)(8 + f), e - 10)", "ldexp((double)(8 + f), e - 9)"),
    ("e4m3_ties_to_odd", "if (d < best_d || (d == best_d && (c & 1) == 0)) {",
     "if (d < best_d || (d == best_d && (c & 1) == 1)) {"),
    ("fp8_store_scale_not_inverted", "float kinv = 1.0f / k_scale[h], vinv = 1.0f / v_scale[h];",
     "float kinv = k_scale[h], vinv = v_scale[h];"),
    ("fp8_decode_v_scale_from_k", "(orc_e4m3_to_double(v[d]) * v_scale[kvh])",
     "(orc_e4m3_to_double(v[d]) * k_scale[kvh])"),
]

PIN_CHECKS = [
    lambda: pins.test_all_16bit_patterns_decode_like_torch(oracle.F16, pins.torch.float16),
    lambda: pins.test_all_16bit_patterns_decode_like_torch(oracle.BF16, pins.torch.bfloat16),
    pins.test_store_then_gather_returns_the_token,
    pins.test_copy_blocks_brute_force,
    pins.test_kv_pack_closed_form,
    pins.test_e4m3_codes_decode_like_torch,
    pins.test_e4m3_encode_round_trip_ties_and_saturation,
    pins.test_fp8_store_matches_torch_quantisation,
    pins.test_fp8_decode_reduces_to_bf16_decode,
    pins.test_kv_pack_unpack_moves_blocks_between_pools,
    pins.test_decode_matches_brute_force_tiny,
    pins.test_decode_matches_brute_force_bf16_gqa_variants,
    pins.test_ctx1_returns_v_exactly,
    lambda: pins.test_split_partitions_merge_to_unsplit(48),
    pins.test_prefill_matches_brute_force,
    pins.test_prefill_special_cases_reduce_to_decode,
]


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutant {name}: anchor text not found exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    str(path), "-o", str(lib), "-lm"], check=True)
    return str(lib)


def run_checks(lib_path: str) -> int:
    """Run every pin check against the oracle build at ``lib_path``; the number
    of checks that reject it."""
    oracle.swap_library(lib_path)
    caught = 0
    for chk in PIN_CHECKS:
        try:
            chk()
        except (AssertionError, ValueError):
            caught += 1
    return caught


def _child(lib_path: str) -> subprocess.CompletedProcess:
    # A mutant may write out of bounds, so each one runs in its own process;
    # a crash counts as caught.
    code = ("import sys; from tests import test_oracle_mutants as m; "
            f"sys.exit(1 if m.run_checks({lib_path!r}) else 0)")
    return subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True,
                          timeout=600)


def test_pins_reject_every_mutant(tmp_path):
    libs = {name: _build_mutant(tmp_path, name, old, new) for name, old, new in MUTANTS}
    with ThreadPoolExecutor(max(1, min(8, os.cpu_count() or 1))) as ex:
        res = dict(zip(libs, ex.map(_child, libs.values())))
    missed = [n for n, r in res.items() if r.returncode == 0]
    assert not missed, f"no pin rejects the planted mistakes {missed}"


def test_unmutated_copy_passes_every_check(tmp_path):
    lib = _build_mutant(tmp_path, "identity", "enum { ORC_F16 = 0, ORC_BF16 = 1 };",
                        "enum { ORC_F16 = 0, ORC_BF16 = 1 };")
    r = _child(lib)
    assert r.returncode == 0, r.stderr.decode()[-2000:]
