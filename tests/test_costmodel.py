"""The cost model of the blocked schedule against the figures the page prints."""
import json
import os

import pytest

from gdn_chunkwise_ut_gb300 import costmodel as cm

with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "paper_counts.json")) as f:
    P = json.load(f)


@pytest.mark.parametrize("C", [32, 64, 128])
def test_blocked_counts(C):
    assert cm.blocked_fma(C) == P["blocked_fma"]["values"][str(C)]
    assert cm.blocked_chain(C) == P["blocked_chain"]["values"][str(C)]
    assert cm.levels(C) == P["recursion_levels"]["values"][str(C)]
    assert C // cm.BASE == P["diag_blocks"]["values"][str(C)]
    assert sum(p for _, p in cm.coupling_pairs(C)) == P["coupling_pairs"]["values"][str(C)]
    assert cm.row_chain(C) == P["row_method_chain"]["values"][str(C)]


def test_row_and_flat_counts():
    assert cm.row_fma(16) == P["diag16_fma"]["value"]
    for C in (32, 64):
        assert cm.row_fma(C) == P["row_method_fma"]["values"][str(C)]
    assert cm.flat_block_fma(64) == P["flat_block_fma_c64"]["value"]
    assert cm.flat_block_gemms(64) == 16
    for C in (64, 128):
        assert cm.flat_block_chain(C) == P["flat_block_chain"]["values"][str(C)]


def test_stage_table_c64():
    assert [list(r) for r in cm.stage_table(64)] == P["stage_widths_c64"]["values"]


@pytest.mark.parametrize("C", [32, 64, 128])
def test_per_token(C):
    f = P["fma_per_token"]
    assert cm.blocked_fma(C) // C == f["values"][str(C)]
    main = cm.main_gemm_per_token(C, 128, 128)
    assert main == f["main_gemm_per_token"][str(C)]
    # the page's share is inverse / (main + inverse), rounded to one decimal
    share = 100 * (cm.blocked_fma(C) / C) / (main + cm.blocked_fma(C) / C)
    assert abs(share - f["inverse_share_percent"][str(C)]) < 0.05 + 1e-9
    # fp16 T write-back: 2C bytes per token (the fp32 T_out here is twice that)
    assert 2 * C == P["t_writeback_bytes_per_token_fp16"]["values"][str(C)]


def test_bytes_per_unit():
    assert cm.bytes_per_unit(64, 128, 128) == 1284
    assert cm.bytes_per_unit(32, 128, 128) == 1156
    assert cm.bytes_per_unit(128, 128, 128) == 1540
    assert cm.bytes_per_unit(64, 128, 128, t_out=False) == 1028  # W and U~ only
    assert cm.bytes_per_unit(64, 128, 128, t_bytes=2) == 1028 + 128  # T in fp16
    assert cm.bytes_per_unit(64, 128, 128, gated=True) == 1284 + 4  # the log decay g
    assert cm.bytes_written_per_unit(64, 128, 128) == 768
    assert cm.bytes_per_unit(32, 64, 64, io_bytes=4) == 1156


def test_not_power_of_two():
    with pytest.raises(ValueError):
        cm.levels(48)
