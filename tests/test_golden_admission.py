"""The host page allocator against the page counts the admission figure prints
(tests/golden/admission_pages.txt): a 2,662-token request on 32-token pages
reserves 86 pages, a short call 5 (prompt and answer reserved together)."""
import os

import pytest

import paged_kv_continuous_pa_gb300 as pa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "admission_pages.txt")


def golden_rows():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            P, prompt, pages = line.split()
            rows.append((int(P), None if prompt == "-" else int(prompt), int(pages)))
    return rows


@pytest.fixture(scope="module", autouse=True)
def lib():
    pa.load()


def test_fixture_is_the_printed_figure():
    assert golden_rows() == [(32, 2662, 86), (32, None, 5)]


@pytest.mark.parametrize("row", golden_rows())
def test_printed_counts_are_reachable_reservations(row):
    P, prompt, pages = row
    if prompt is None:
        # every request of 4 * 32 + 1 .. 5 * 32 tokens (prompt + answer) takes 5 pages, no other does
        for total in range(1, 8 * P):
            assert (pa.pages_needed(P, total, 0) == pages) == (4 * P < total <= 5 * P)
            assert pa.pages_needed(P, total // 2, total - total // 2) == pa.pages_needed(P, total, 0)
        return
    assert pa.pages_needed(P, prompt, 0) == 84 < pages  # the prompt alone does not explain the count
    budgets = [a for a in range(0, 4 * P) if pa.pages_needed(P, prompt, a) == pages]
    # answer budgets of 59 .. 90 tokens give the printed 86 pages: ceil((2662 + a) / 32) == 86
    assert budgets == list(range(59, 91))
    a = pa.Pages(num_pages=100, page_size=P, num_seqs=1, max_blocks=90)
    st, info = a.admit(0, prompt, budgets[-1])
    assert st == pa.PA_OK and info.pages_needed == pages
    assert int((a.block_tables[0] >= 0).sum()) == pages and a.free_count() == 100 - pages


def test_one_token_more_than_the_printed_reservation_needs_another_page():
    a = pa.Pages(num_pages=86, page_size=32, num_seqs=2, max_blocks=90)
    st, info = a.admit(0, 2662, 91)  # 2753 tokens: 87 pages, 86 exist
    assert st == pa.PA_ERR_NO_PAGES and (info.pages_needed, info.pages_free) == (87, 86)
    st, info = a.admit(0, 2662, 90)
    assert st == pa.PA_OK and a.free_count() == 0
