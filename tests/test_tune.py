"""Host logic of the route-block tuning: the paired gate (>= 1 % median paired
improvement and >= 25/31 faster pairs), the CSV table round trip and the
bucket lookup MoeLayer applies."""
import types

import pytest

from block_scaled_moe_sort_gb300 import MoeLayer
from block_scaled_moe_sort_gb300 import tune


def test_gate_adopts_a_consistent_two_percent_win():
    base = [100.0] * 31
    cand = [98.0] * 31
    g = tune.paired_gate(base, cand)
    assert g["accept"] and g["wins"] == 31 and abs(g["median_gain"] - 0.02) < 1e-12


def test_gate_thresholds_are_inclusive():
    # exactly 25 of 31 faster pairs, median gain exactly 1 %
    base = [100.0] * 31
    cand = [99.0] * 25 + [100.5] * 6
    g = tune.paired_gate(base, cand)
    assert g["wins"] == 25 and g["wins_needed"] == 25
    assert abs(g["median_gain"] - 0.01) < 1e-12 and g["accept"]


def test_gate_rejects_too_few_wins_even_with_a_large_median():
    base = [100.0] * 31
    cand = [90.0] * 24 + [101.0] * 7
    g = tune.paired_gate(base, cand)
    assert g["median_gain"] > 0.05 and g["wins"] == 24 and not g["accept"]


def test_gate_rejects_a_small_gain():
    base = [100.0] * 31
    cand = [99.5] * 31
    assert not tune.paired_gate(base, cand)["accept"]


def test_gate_rejects_identical_measurements():
    xs = [100.0 + i * 0.01 for i in range(31)]
    g = tune.paired_gate(xs, list(xs))
    assert g["wins"] == 0 and g["median_gain"] == 0 and not g["accept"]


def test_gate_needs_paired_lists():
    with pytest.raises(ValueError):
        tune.paired_gate([1.0, 2.0], [1.0])
    with pytest.raises(ValueError):
        tune.paired_gate([], [])


def test_gate_scales_the_win_count_with_the_pairs():
    g = tune.paired_gate([100.0] * 62, [98.0] * 50 + [101.0] * 12)
    assert g["wins_needed"] == 50 and g["accept"]


def _row(max_tokens, bm, H=5120, Ip=640, E=384, topk=6, a16=0):
    return {"H": H, "Ip": Ip, "E": E, "topk": topk, "a16": a16, "max_tokens": max_tokens,
            "block_m": bm, "default_block_m": 16, "median_gain": 0.02, "wins": 30,
            "pairs": 31, "control_gain": 0.0, "control_wins": 15}


def test_table_round_trip_and_geometry_filter(tmp_path):
    rows = [_row(64, 32), _row(8, 16), _row(1024, 64), _row(16, 16, E=128, topk=3)]
    p = tmp_path / "t.csv"
    tune.write_table(rows, str(p))
    back = tune.read_table(str(p))
    assert [{k: r[k] for k in rows[0]} for r in back] == rows
    assert all(r["prefetch1"] == 0 and r["prefetch2"] == 0 for r in back)   # knob unset
    assert tune.table_for(back, 5120, 640, 384, 6, False) == [(8, 16), (64, 32), (1024, 64)]
    assert tune.table_for(back, 5120, 640, 128, 3, False) == [(16, 16)]
    assert tune.table_for(back, 5120, 640, 384, 6, True) == []


def test_layer_bucket_lookup():
    # MoeLayer.block_m_for only reads block_m_table (no GPU needed)
    lay = types.SimpleNamespace(block_m_table=[(8, 16), (64, 32), (1024, 64)])
    f = MoeLayer.block_m_for
    assert [f(lay, M) for M in (1, 8, 9, 64, 65, 1024)] == [16, 16, 32, 32, 64, 64]
    assert f(lay, 1025) == 0                      # beyond the table: library rule
    assert f(types.SimpleNamespace(block_m_table=[]), 5) == 0


def test_shipped_table_is_consistent_with_the_gate():
    rows = tune.read_table(tune.PACKAGED_TABLE)
    assert rows
    for r in rows:
        assert r["block_m"] in (16, 32, 64, 128, 256)
        assert r["pairs"] == 31
        if r["block_m"] != r["default_block_m"]:
            # adopted rows passed the gate
            assert r["median_gain"] >= tune.MIN_GAIN and r["wins"] >= 25
        # no identical-configuration control passed it
        assert not (r["control_gain"] >= tune.MIN_GAIN and r["control_wins"] >= 25)
    # both geometries the pages tune, with their eight token buckets
    for E, k in ((384, 6), (128, 3)):
        buckets = [b for b, _ in tune.packaged_table_for(5120, 640, E, k, False)]
        assert buckets == [8, 16, 32, 64, 128, 256, 512, 1024]


def test_layer_lookup_by_topk_for_shipped_rows():
    lay = types.SimpleNamespace(block_m_table=[],
                                _bm_by_topk={3: [(512, 16), (1024, 32)], 6: [(1024, 16)]})
    f = MoeLayer.block_m_for
    assert f(lay, 640, 3) == 32 and f(lay, 640, 6) == 16 and f(lay, 640, 4) == 0


def test_shipped_rows_by_geometry():
    from block_scaled_moe_sort_gb300 import shipped_block_m_rows
    draft = shipped_block_m_rows(5120, 640, 128, False)
    # rows: (max_tokens, block_m[, prefetch1, prefetch2[, split]])
    assert list(draft) == [3] and draft[3][-1][:2] == (1024, 32)
    backbone = shipped_block_m_rows(5120, 640, 384, False)
    assert [r[1] for r in backbone[6]] == [16] * 8
    # the weight prefetch leads: against the short defaults (4 / 2) only the
    # bucket 16 row passed the gate (2 / 2)
    pf = lambda rows: {r[0]: (tuple(r[2:4]) if len(r) >= 4 else (0, 0)) for r in rows}
    assert pf(backbone[6])[16] == (2, 2)
    assert set(pf(backbone[6]).values()) == {(0, 0), (2, 2)}
    # the split walk is the library's choice; whole tiles only won at one
    # draft bucket (16)
    split = lambda rows: {r[0]: (r[4] if len(r) == 5 else 0) for r in rows}
    assert set(split(backbone[6]).values()) == {0}
    assert split(draft[3]) == {8: 0, 16: 2, 32: 0, 64: 0, 128: 0, 256: 0, 512: 0, 1024: 0}
    bm = lambda rows: {r[0]: r[1] for r in rows}
    # expert-parallel shard (96 local experts of 384, routing over all 384)
    ep = shipped_block_m_rows(5120, 2304, 96, False)
    assert list(ep) == [6] and ep[6][-1] == (16384, 128)          # prefill: defaults kept
    assert bm(ep[6])[32] == 32 and bm(ep[6])[2048] == 64
    assert set(split(ep[6]).values()) == {0}
    # a16w4: 384 top-6, and 385 top-7 with the shared expert as expert 384;
    # no prefetch lead and no split setting passed the gate (the converters
    # bound these calls)
    a16 = shipped_block_m_rows(5120, 768, 384, True)
    assert list(a16) == [6] and bm(a16[6])[1024] == 32 and bm(a16[6])[4096] == 128
    assert all(len(r) == 2 for r in a16[6])
    assert list(shipped_block_m_rows(5120, 768, 385, True)) == [7]
    assert shipped_block_m_rows(4096, 640, 384, False) == {}     # not tuned
    lay = types.SimpleNamespace(block_m_table=[], _bm_by_topk=draft)
    assert MoeLayer.block_m_for(lay, 640, 3) == 32 and MoeLayer.block_m_for(lay, 320, 3) == 16
    assert MoeLayer.prefetch_for(lay, 640, 3) == pf(draft[3])[1024] == (0, 0)
    assert MoeLayer.split_for(lay, 10, 3) == 2 and MoeLayer.split_for(lay, 640, 3) == 0


def test_prefetch_knob_round_trip_and_lookup(tmp_path):
    rows = [_row(64, 32), _row(1024, 64)]
    rows[1].update(prefetch1=24, prefetch2=4, prefetch_gain=0.02, prefetch_wins=30)
    p = tmp_path / "t.csv"
    tune.write_table(rows, str(p))
    back = tune.read_table(str(p))
    assert back[0]["prefetch1"] == 0 and back[0]["prefetch2"] == 0
    assert (back[1]["prefetch1"], back[1]["prefetch2"], back[1]["prefetch_wins"]) == (24, 4, 30)
    # a table written before the knob existed reads with zeros
    old = tmp_path / "old.csv"
    old.write_text("H,Ip,E,topk,a16,max_tokens,block_m,default_block_m,median_gain,wins,pairs,"
                   "control_gain,control_wins\n5120,640,384,6,0,8,16,16,0.0,0,31,0.0,15\n")
    r = tune.read_table(str(old))[0]
    assert (r["prefetch1"], r["prefetch2"], r["prefetch_gain"]) == (0, 0, 0.0)
    lay = types.SimpleNamespace(block_m_table=[(64, 32), (1024, 64, 24, 4)])
    assert MoeLayer.block_m_for(lay, 10) == 32 and MoeLayer.prefetch_for(lay, 10) == (0, 0)
    assert MoeLayer.block_m_for(lay, 500) == 64 and MoeLayer.prefetch_for(lay, 500) == (24, 4)
    assert MoeLayer.prefetch_for(lay, 5000) == (0, 0)


def test_split_knob_round_trip_and_lookup(tmp_path):
    # the third knob: split walk 0 (rule) / 1 (always) / 2 (never); a row
    # that sets it carries the prefetch leads too (0 = defaults)
    rows = [_row(64, 32), _row(1024, 64)]
    rows[1].update(split=1, split_gain=0.04, split_wins=31)
    p = tmp_path / "t.csv"
    tune.write_table(rows, str(p))
    back = tune.read_table(str(p))
    assert (back[0]["split"], back[0]["split_gain"], back[0]["split_wins"]) == (0, 0.0, 0)
    assert (back[1]["split"], back[1]["split_gain"], back[1]["split_wins"]) == (1, 0.04, 31)
    lay = types.SimpleNamespace(block_m_table=[(64, 32), (1024, 64, 0, 0, 1), (4096, 64, 8, 2)])
    assert MoeLayer.split_for(lay, 10) == 0 and MoeLayer.prefetch_for(lay, 10) == (0, 0)
    assert MoeLayer.split_for(lay, 500) == 1 and MoeLayer.prefetch_for(lay, 500) == (0, 0)
    assert MoeLayer.split_for(lay, 2000) == 0 and MoeLayer.prefetch_for(lay, 2000) == (8, 2)
    assert MoeLayer.split_for(lay, 5000) == 0
