"""Size-law pins: the oracle's byte arithmetic against numbers the pages print.

Sources: trefon.com "Matematyka cache KV" (sections "Bajty na token",
"Przyklad: model 27B przy 262K" and its format table); nalar.dev "Kuantisasi KV
Cache dengan Error Budget yang Eksplisit" (section "Ukuran cache mengikuti
jumlah elemen tersimpan dan bit width"); troisinh.com "KV Cache Quantization"
(opening paragraph and section "Van de").
"""

import os

import pytest

from oracle import kvq_oracle as O

KiB, MiB, GiB = 1 << 10, 1 << 20, 1 << 30


def _read_table(golden_dir, name):
    rows = []
    with open(os.path.join(golden_dir, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _read_kv(golden_dir, name):
    out = {}
    for r in _read_table(golden_dir, name):
        out[r[0]] = float(r[1])
    return out


def _parse_size(s):
    for unit, mult in (("GiB", GiB), ("MiB", MiB)):
        if s.endswith(unit):
            return float(s[: -len(unit)]), mult
    raise ValueError(s)


def _model_32768(fmt):
    # 16 layers x 4 kv heads x D=256: 2*16*4*256 = 32,768 cached values per token.
    return O.Config(L=16, H_kv=4, H_q=24, D=256, batch=1, max_T=262144, k_fmt=fmt, v_fmt=fmt)


def test_block_bytes_match_named_layouts():
    # trefon.com format table: Q8_0 34 B/32, Q4_0 18 B/32, TBQ4 66 B/128, 3-bit 50 B/128.
    assert O.block_bytes(8, 32) == 34
    assert O.block_bytes(4, 32) == 18
    assert O.block_bytes(4, 128) == 66
    assert O.block_bytes(3, 128) == 50
    # the same law for the 2-bit cold tier: fp16 scale + 32*2/8 bytes
    assert O.block_bytes(2, 32) == 10


def test_scalar_count_formula():
    # nalar.dev: 2 * L * T * H_kv * D scalars; the 2 is key plus value.
    assert O.scalars(L=1, T=1, H_kv=1, D=1) == 2
    assert O.scalars(L=32, T=10, H_kv=32, D=128) == 2 * 32 * 10 * 32 * 128


def test_format_table_every_cell(golden_dir):
    rows = _read_table(golden_dir, "format_table_262k.txt")
    assert len(rows) == 5
    for name, bits, group, bpv, per_tok_kib, *sizes in rows:
        fmt = O.Fmt(int(bits), int(group))
        cfg = _model_32768(fmt)
        # bits per value column
        assert O.block_bytes(fmt.bits, fmt.group) * 8 / fmt.group == pytest.approx(float(bpv))
        # per-token column (exact)
        assert O.bytes_per_token(cfg) == float(per_tok_kib) * KiB
        # the four context columns, to the page's printed rounding
        for T, printed in zip((8192, 32768, 131072, 262144), sizes):
            val, unit = _parse_size(printed)
            got = O.cache_bytes(cfg, T) / unit
            decimals = len(printed.split(".")[1].rstrip("GiMB")) if "." in printed else 0
            tol = 0.5 * 10 ** (-decimals) if decimals else 1e-12
            assert abs(got - val) <= tol + 1e-12, (name, T, got, printed)


def test_27b_worked_example(golden_dir):
    kv = _read_kv(golden_dir, "size_law_worked.txt")
    cache = kv["tbq4_cache_mib_at_262144"] * MiB
    per_token = cache / 262144
    assert per_token == kv["tbq4_bytes_per_token"]
    assert per_token / 66 * 128 == kv["values_per_token"]
    # and the forward direction through the oracle's size law
    cfg = _model_32768(O.Fmt(4, 128))
    assert O.cache_bytes(cfg, 262144) == 4224 * MiB
    assert O.bytes_per_token(cfg) == 16896
    assert O.scalars(cfg.L, 1, cfg.H_kv, cfg.D) == 32768
    # the 3-bit layout on the same model
    cfg3 = _model_32768(O.Fmt(3, 128))
    assert O.cache_bytes(cfg3, 262144) == 3200 * MiB


def test_24gb_card_budget(golden_dir):
    kv = _read_kv(golden_dir, "size_law_worked.txt")
    budget = kv["budget_gib"] * GiB
    fp16 = budget // O.bytes_per_token(_model_32768(O.Fmt(16, 128)))
    q8 = budget // O.bytes_per_token(_model_32768(O.Fmt(8, 32)))
    four = budget // O.bytes_per_token(_model_32768(O.Fmt(4, 128)))
    assert fp16 == 114688 and abs(fp16 - kv["fp16_tokens_approx"]) / kv["fp16_tokens_approx"] < 0.05
    assert q8 == 215883 and abs(q8 - kv["q8_0_tokens_approx"]) / kv["q8_0_tokens_approx"] < 0.05
    assert four >= kv["four_bit_min_tokens"]


def test_llama_sizes(golden_dir):
    kv = _read_kv(golden_dir, "size_law_worked.txt")
    # Llama-2-7B: 32 layers, 32 kv heads, head dim 128, fp16
    llama7 = O.Config(L=32, H_kv=32, H_q=32, D=128, batch=1, max_T=1, k_fmt=O.Fmt(16, 128), v_fmt=O.Fmt(16, 128))
    bpt = O.bytes_per_token(llama7)
    assert bpt == 524288 == O.scalars(32, 1, 32, 128) * 2
    assert abs(bpt * 10_000 / 1e9 - kv["llama2_7b_gb_at_10k_approx"]) < 0.5
    assert bpt * 100_000 / 1e9 > kv["llama2_7b_gb_at_100k_min"]
    assert bpt * 1_000_000 / 1e9 > kv["llama2_7b_gb_at_1m_min"]
    # LLaMA-70B: 80 layers, 8 kv heads (GQA), head dim 128
    llama70 = O.Config(L=80, H_kv=8, H_q=64, D=128, batch=1, max_T=1, k_fmt=O.Fmt(16, 128), v_fmt=O.Fmt(16, 128))
    assert O.bytes_per_token(llama70) * 1_000_000 / 1e9 > kv["llama_70b_gb_at_1m_min"]


def test_cache_bytes_counts_window_and_tiers():
    # KIVI 4-bit with a 128-token 16-bit window: at T = 32768 the quantized
    # prefix is 32640 tokens and the window exactly 128.
    cfg = O.Config(L=32, H_kv=32, H_q=32, D=128, batch=1, max_T=32768,
                   k_fmt=O.Fmt(4, 32, O.AXIS_CHANNEL), v_fmt=O.Fmt(4, 32), residual_window=128)
    assert O.q_end(cfg, 32768) == 32640
    per_head = 32640 // 32 * 128 * 18 + 32640 * 4 * 18 + 2 * 128 * 128 * 2
    assert O.cache_bytes(cfg, 32768) == 32 * 32 * per_head
    # hot/cold split of the Mistral-7B-shaped workload
    cfg5 = O.Config(L=32, H_kv=8, H_q=32, D=128, batch=64, max_T=32768,
                    k_fmt=O.Fmt(4, 32, O.AXIS_CHANNEL), v_fmt=O.Fmt(4, 32),
                    k_cold=O.Fmt(2, 32, O.AXIS_CHANNEL), v_cold=O.Fmt(2, 32),
                    hot_window=4096, residual_window=128)
    assert (O.c_end(cfg5, 32768), O.q_end(cfg5, 32768)) == (28544, 32640)
    per_head = (28544 // 32 * 128 * 10 + 28544 * 4 * 10) + (4096 // 32 * 128 * 18 + 4096 * 4 * 18) + 2 * 128 * 128 * 2
    assert O.cache_bytes(cfg5, 32768) == 32 * 8 * per_head
    # steady state counts the cold format
    assert O.bytes_per_token(cfg5) == 32 * 8 * (40 + 40)
