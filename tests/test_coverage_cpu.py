"""The full-size GPU parity tests compare a row sample, not every row; these CPU
checks pin what that sample covers. Work items are (query tile, KV group):
21-token tiles for the one-CTA kernel, 42-token tiles for the CTA pair. The
sample must hold a row of every item and a row of every item's last token (the
row every KV piece of a split item contributes to), at every workload size."""
import numpy as np
import pytest

from gqa_inputs import WORKLOADS, sample_rows
from tests.gpu_helpers import item_cover_rows, unchecked_items


@pytest.mark.parametrize("q_len", [1, 2, 20, 21, 22, 41, 42, 43, 127, 128, 129] +
                         sorted({w.q_len for w in WORKLOADS.values()}))
@pytest.mark.parametrize("tpi", [21, 42])
def test_cover_rows_check_every_item(q_len, tpi):
    rows = item_cover_rows(q_len, 24)
    assert rows.min() >= 0 and rows.max() < q_len * 24
    assert unchecked_items(rows, q_len, tpi) == []


def test_counting_finds_a_missing_item():
    rows = item_cover_rows(4096, 24)
    tok, head = rows // 24, rows % 24
    drop = (tok // 42 == 17) & (head // 6 == 2)  # every row of pair item (17, 2)
    assert unchecked_items(rows[~drop], 4096, 42) == [(17, 2)]
    last = (tok == 42 * 17 + 41) & (head // 6 == 2)  # only that item's last-token rows
    assert unchecked_items(rows[~last], 4096, 42) == [(17, 2)]


def test_stratified_sample_alone_misses_items():
    """Why the cover rows exist: 1200 stratified rows of a 4096-token chunk leave
    most items without their last token."""
    rows = sample_rows(4096, 24, 1200, seed=5).numpy()
    assert len(unchecked_items(rows, 4096, 21)) > 700
    assert unchecked_items(item_cover_rows(4096, 24, rows), 4096, 21) == []
