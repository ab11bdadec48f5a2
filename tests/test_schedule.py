"""The binding's schedule choice (host logic, no GPU): "auto" takes the
one-head kernel for gated 128 x 128 calls (with or without mean correction)
and the paired kernel otherwise; the 128 x 224 tile has only the one-head
kernel."""
import pytest

from block_sparse_gated_gb300.api import resolve_schedule


@pytest.mark.parametrize("mode", ["threshold", "lambda"])
def test_auto_takes_pipelined_for_gated_128(mode):
    assert resolve_schedule("auto", mode=mode) == "pipelined"
    assert resolve_schedule("auto", mode=mode, mean_correction=True) == "pipelined"


@pytest.mark.parametrize("kw", [dict(mode="none"), dict(block_q=64), dict(block_k=64),
                                dict(block_q=64, block_k=64)])
def test_auto_takes_paired_elsewhere(kw):
    args = dict(mode="threshold")
    args.update(kw)
    assert resolve_schedule("auto", **args) == "paired"


def test_explicit_choice_is_kept():
    assert resolve_schedule("paired", mode="threshold") == "paired"
    assert resolve_schedule("pipelined", mode="none") == "pipelined"


def test_tile224_is_one_head():
    assert resolve_schedule("auto", block_k=224) == "pipelined"
    assert resolve_schedule("paired", block_k=224) == "pipelined"


def test_unknown_schedule_raises():
    with pytest.raises(ValueError):
        resolve_schedule("fast")
