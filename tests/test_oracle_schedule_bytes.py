"""Pins of the oracle's layer-type map, IndexCache schedule and byte accounting
against the values the pages print (tests/golden/*.txt)."""
import os

import numpy as np
import pytest

import oracle
from deepseek_v4_compressed_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.split() for l in f if l.strip() and not l.startswith("#")]


def test_layer_types_match_pages():
    for ratio, expect in golden_lines("layer_types.txt"):
        assert oracle.layer_type(int(ratio)) == int(expect)


def test_indexcache_freq2_reproduces_page_schedule():
    gold = {l[0]: l[1:] for l in golden_lines("indexcache_freq2.txt")}
    ratios = synth.mixed_stack_ratios()
    assert len(ratios) == 60
    c4 = np.nonzero(ratios == 4)[0]
    assert len(c4) == int(gold["c4_layers"][0])
    skip = oracle.index_schedule(ratios, True, 2)
    assert int(skip.sum()) == int(gold["reuse"][0])
    assert len(c4) - int(skip.sum()) == int(gold["compute"][0])
    assert list(np.nonzero(skip)[0]) == [int(x) for x in gold["skip_layer_ids"]]
    assert np.all(skip[ratios != 4] == 0)


def test_indexcache_freq1_and_off_skip_nothing():
    ratios = synth.mixed_stack_ratios()
    assert not oracle.index_schedule(ratios, True, 1).any()
    assert not oracle.index_schedule(ratios, False, 2).any()


def test_indexcache_pattern_precedence():
    ratios = np.array([4, 1, 4, 4, 128, 4, 4, 4], np.int32)   # c4 rank: 0,_,1,2,_,3,4,5
    skip = oracle.index_schedule(ratios, True, 2, pattern="FSS")
    # pattern wins over freq 2; ranks past the string compute
    assert list(skip) == [0, 0, 1, 1, 0, 0, 0, 0]
    skip = oracle.index_schedule(ratios, True, 2, pattern="F")
    assert not skip.any()
    assert oracle.index_schedule(ratios, True, 2, pattern="SF") is None
    assert oracle.index_schedule(ratios, True, 2, pattern="FX") is None
    assert oracle.index_schedule(ratios, True, 0) is None


def test_entry_bytes_match_pages():
    for kind, dim, nbytes in (l for l in golden_lines("kv_bytes.txt") if l[0].endswith("entry")):
        if kind == "idx_entry":
            assert oracle.idx_entry_bytes(int(dim)) == int(nbytes)
        else:
            assert oracle.mla_entry_bytes(int(dim), 64) == int(nbytes)


def test_block_table_and_total_match_pages():
    rows = [l for l in golden_lines("kv_bytes.txt") if l[0] == "block"]
    fp8_entry = {"c4_indexer": oracle.idx_entry_bytes(128),
                 "c4_attention": oracle.mla_entry_bytes(448, 64),
                 "c128_attention": oracle.mla_entry_bytes(448, 64)}
    per_token_fp16 = {}
    for _, name, entries, dims, fp16_b, fp8_b in rows:
        entries, dims = int(entries), int(dims)
        assert entries * dims * 2 == int(fp16_b)
        assert entries * fp8_entry[name] == int(fp8_b)
        per_token_fp16[name] = entries * dims * 2 / 256
    c4a = per_token_fp16["c4_indexer"] + per_token_fp16["c4_attention"]
    c128a = per_token_fp16["c128_attention"]
    assert (c4a, c128a) == (320, 8)
    total_mib = (30 * c4a + 31 * c128a) * 2 ** 20 / 2 ** 20
    gold_total = int([l for l in golden_lines("kv_bytes.txt") if l[0] == "total_mib"][0][1])
    assert total_mib == gold_total
    assert total_mib / 1024 == pytest.approx(9.6171875)
