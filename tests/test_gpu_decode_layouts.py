"""The hybrid decode's two shared-memory layouts -- the ordinary one (one 16-token unit of K / V
rows staged per warp at a time, summary rows read straight from global memory) and the wide one
(every kept summary row staged at once, every selected token staged per warp at once) -- each
checked against the oracle on the same cases. The launch takes the wide layout only when every
(unit, KV head) has an SM of its own; the test hook of include/rkv_testing.h forces either."""
import pytest

from tests import test_gpu_decode as T

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[1, 2], ids=["ordinary", "wide"])
def layout(request):
    rkv = T._lib()
    rkv.rkv_testing_decode_layout(request.param)
    yield request.param
    rkv.rkv_testing_decode_layout(0)


def test_layout_config1_shape(layout):
    T.test_hybrid_config1_shape()


def test_layout_ragged_and_dense(layout):
    T.test_hybrid_ragged_and_dense_fallback()


@pytest.mark.parametrize("gqa", [1, 8])
def test_layout_gqa(layout, gqa):
    T.test_hybrid_gqa_variants(gqa)


@pytest.mark.parametrize("budget,page,channels", [(1024, 4, 32), (256, 16, 128), (128, 1, 16)])
def test_layout_budget_page_channels(layout, budget, page, channels):
    T.test_hybrid_budget_page_channel_variants(budget, page, channels)


def test_layout_two_rounds_of_page_groups(layout):
    # 2112 pages: the ordinary layout's thread pairs take a second round of 8-page groups (264
    # groups for 128 pairs); the wide layout stages them all at once
    T._hybrid_case(2, 2, 4, [8448, 8001], 8448, 512, 4, 32, seed=71, steps=2)


def test_layout_general_select(layout):
    # 5001 pages: beyond the register-resident select (and the wide layout's shared memory,
    # so both runs take the ordinary layout)
    T.test_hybrid_more_than_4096_pages_general_select()


def test_layout_append_steps(layout):
    T.test_hybrid_append_steps()


def test_layout_more_units_than_sms(layout):
    # 160 (unit, KV head) pairs, more than the SMs: the wide layout runs here only when forced
    T._hybrid_case(80, 2, 4, [600 + 7 * i for i in range(80)], 1200, 256, 4, 32, seed=73,
                   steps=1)
