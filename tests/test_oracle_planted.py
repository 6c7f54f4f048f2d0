"""Planted mistakes: the pins must reject a wrong oracle.

Each case below alters one expression of ``oracle/oracle.cpp`` the way a
plausible slip would (a dropped term, a wrong sign, index or operand, an
off-by-one, the wrong rounding), builds the altered copy into a temporary
library, and runs the oracle's pins (``test_oracle_pins.py``) and the cases
worked by hand (``test_golden.py``) against it in a child pytest
(``DS_ORACLE_LIB`` points the loader at the copy). The child must report a
failed test: a mistake that every pin lets through would mean the oracle is
not pinned where that mistake sits. Everything runs on the CPU; every altered
copy keeps its memory accesses inside the buffers the pins pass.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.cpp")

# name -> (exact text in oracle.cpp, its replacement)
PLANTED = {
    # stage 1: proxy scores
    "score_channel_reversed": ("label[(slot * HL + gL) * C + c]", "label[(slot * HL + gL) * C + (C - 1 - c)]"),
    "score_sum_dropped": ("s += qv * lv;", "s = qv * lv;"),
    "score_label_head_always_0": ("const int gL = (HL == 1) ? 0 : g;", "const int gL = 0;"),
    "score_group_interleaved": ("for (int h = g * G; h < (g + 1) * G; ++h) {\n          for (int c = 0; c < C; ++c) {",
                                "for (int h = g; h < Hq; h += Hkv) {\n          for (int c = 0; c < C; ++c) {"),
    "slot_offset_by_one": ("return page * page_size + t % page_size;", "return page * page_size + (t + 1) % page_size;"),
    # stage 2: top-k
    "topk_ties_to_higher_index": ("return x < y;                        // equal scores",
                                  "return x > y;                        // equal scores"),
    "topk_nan_ranks_first": ("if (nx != ny) return ny;             // a number",
                             "if (nx != ny) return nx;             // a number"),
    "topk_output_unsorted": ("std::vector<int32_t> chosen(order.begin(), order.begin() + keff);\n"
                             "      std::sort(chosen.begin(), chosen.end());",
                             "std::vector<int32_t> chosen(order.begin(), order.begin() + keff);"),
    "sharded_local_topk_short": ("const int kj = std::min(k, static_cast<int>(local.size()));",
                                 "const int kj = std::min(k / 2 + 1, static_cast<int>(local.size()));"),
    # stage 3: attention
    "attn_scale_dropped": ("z[i] = sm_scale * dot;", "z[i] = dot;"),
    "attn_value_is_key": ("o[d] += w * vval(slot, g, d);", "o[d] += w * kval(slot, g, d);"),
    "attn_lse_without_max": ("lse = m + std::log(l);", "lse = std::log(l);"),
    "attn_v_uses_k_scale": ("(v_cache)[e]) * v_scale[slot / page_size];", "(v_cache)[e]) * k_scale[slot / page_size];"),
    "split_pages_by_token": (": ((row[i] / page_size) % S == j);", ": (row[i] % S == j);"),
    "split_chunks_overlap": ("i < static_cast<long long>(j + 1) * n / S)", "i <= static_cast<long long>(j + 1) * n / S)"),
    # stage 4: merge
    "merge_weight_uses_max": ("const double w = std::exp(lse_part[j * rows + r] - lse[r]);",
                              "const double w = std::exp(lse_part[j * rows + r] - m);"),
    # number formats
    "e4m3_bias_8": ("exp - 7);  // normal", "exp - 8);  // normal"),
    "e4m3_subnormal_exponent": ("1 - 7);        // subnormal", "0 - 7);        // subnormal"),
    "e4m3_ties_to_odd": ("(err == best_err && (c & 1) == 0)", "(err == best_err && (c & 1) == 1)"),
    "bf16_ties_away_from_zero": ("std::nearbyint(std::ldexp(x, -qexp))", "std::round(std::ldexp(x, -qexp))"),
    "bf16_nine_bits": ("std::max(e - 8, -133)", "std::max(e - 9, -133)"),
    # cache append
    "append_label_from_v": ("v = k_new[(static_cast<long long>(b) * Hkv + g) * D + ch];",
                            "v = v_new[(static_cast<long long>(b) * Hkv + g) * D + ch];"),
    "append_fp8_multiplies_scale": ("bf16_value(k_new[src])) / k_scale[page];", "bf16_value(k_new[src])) * k_scale[page];"),
    # block-compressed selection
    "block_mean_over_full_page": ("sum / static_cast<double>(t1 - t0)", "sum / static_cast<double>(page_size)"),
    "block_score_logical_page": ("bf16_value(block_keys[pid * C + c])", "bf16_value(block_keys[j * C + c])"),
    "block_expand_past_length": ("t < (blk[i] + 1LL) * page_size && t < T;", "t < (blk[i] + 1LL) * page_size;"),
}


def _build_and_run(name, old, new, tmpdir):
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: the text to alter must occur exactly once in oracle.cpp"
    cpp = os.path.join(tmpdir, f"{name}.cpp")
    lib = os.path.join(tmpdir, f"lib{name}.so")
    with open(cpp, "w") as f:
        f.write(src.replace(old, new))
    subprocess.check_call([os.environ.get("CXX", "g++"), "-O1", "-std=c++17", "-shared", "-fPIC", "-o", lib, cpp])
    # One thread per child: several children run at once.
    env = dict(os.environ, DS_ORACLE_LIB=lib, OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py"), os.path.join(ROOT, "tests", "test_golden.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode, (r.stdout + r.stderr)[-1500:]


def test_every_planted_mistake_fails_a_pin(tmp_path):
    workers = max(1, min(8, os.cpu_count() or 1))
    with ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda kv: _build_and_run(kv[0], kv[1][0], kv[1][1], str(tmp_path)), PLANTED.items()))
    # pytest exits 1 when a test failed; anything else (0: all passed, a crash) is not a pin's rejection.
    missed = [(name, rc, tail) for name, rc, tail in results if rc != 1]
    assert not missed, "planted mistakes not rejected by a pin:\n" + "\n".join(
        f"--- {name} (exit {rc})\n{tail}" for name, rc, tail in missed)


def test_the_unaltered_oracle_passes_the_same_run(tmp_path):
    # The control: the same child run on an unaltered copy passes, so the
    # failures above come from the planted mistakes.
    name, rc, tail = _build_and_run("control", "return 0;\n}\n\n}  // extern \"C\"", "return 0;\n}\n\n}  // extern \"C\"",
                                    str(tmp_path))
    assert rc == 0, tail
