"""CPU checks of the implicit-im2col convolution's tiling (bt_conv2d_plan_info,
host only): for every plan the planner or the measured selection can take,
the bands cover the output rows with none empty, a tile's accumulator columns
cover its rows of virtual pixels, the staged rows cover every tap's shifted
reach, and shared memory fits one CTA."""
import itertools

import pytest
import torch

import xnor_popcount_gemm_gb300 as bt

GEOMS = [  # B, C, H, W, O, k, s, p, d
    (128, 256, 14, 14, 256, 3, 1, 1, 1),     # the benchmark's stride-1 layer
    (256, 128, 28, 28, 256, 3, 2, 1, 1),     # stride 2
    (256, 128, 28, 28, 256, 3, 2, 2, 2),     # stride 2, dilation 2
    (64, 64, 56, 56, 64, 3, 1, 1, 1),
    (64, 64, 56, 56, 128, 3, 2, 1, 1),
    (256, 512, 7, 7, 512, 3, 1, 1, 1),
    (32, 512, 7, 7, 2048, 1, 1, 0, 1),
    (3, 64, 17, 19, 96, 3, 1, 1, 1),         # odd sizes
    (2, 64, 30, 33, 70, 3, 1, 1, 1),
    (1, 96, 57, 23, 40, 5, 2, 2, 1),         # 5x5
    (2, 64, 11, 11, 48, 7, 1, 3, 1),         # 7x7
    (1, 32, 20, 200, 16, 3, 1, 1, 1),        # wide rows
    (400, 40, 1, 1, 17, 3, 1, 1, 1),         # 1x1 images
    (360, 64, 3, 3, 96, 3, 1, 1, 1),
    (2, 384, 9, 9, 33, 3, 1, 1, 1),          # three 64-byte slices per tap
]


def _out(h, k, s, p, d):
    return (h + 2 * p - d * (k - 1) - 1) // s + 1


@pytest.fixture(autouse=True)
def _no_plan_env(monkeypatch):
    for v in ("BT_CONV_PAIR", "BT_CONV_PLAN", "BT_CONV_FUSED", "BT_CONV_SPLIT", "BT_CONV_IMPLICIT"):
        monkeypatch.delenv(v, raising=False)


@pytest.mark.parametrize("geom", GEOMS)
def test_every_plan_covers_the_output(geom):
    B, C, H, W, O, k, s, p, d = geom
    Ho, Wo = _out(H, k, s, p, d), _out(W, k, s, p, d)
    seen = 0
    for code, od, pair, split in itertools.product((bt.BT_CODE_E4M3, bt.BT_CODE_E2M1), (torch.float32, torch.bfloat16),
                                                   (-1, 0, 1), (1, 2, 4)):
        info = bt.bt_conv2d_plan_info(B, C, H, W, O, k, s, p, d, code, od, 152, pair, split)
        if not info["implicit"]:
            continue
        seen += 1
        bands, ht, ht2, wv = info["bands"], info["band_rows"], info["cta_rows"], info["row_width"]
        n, nb, rv = info["tile_n"], info["cta_n"], info["staged_rows"]
        assert wv >= Wo
        # the bands cover the rows and none is empty
        assert bands * ht >= Ho and (bands - 1) * ht < Ho, info
        if info["pair"]:
            assert ht == 2 * ht2 and n == 2 * nb and nb % 8 == 0 and nb >= ht2 * wv, info
        else:
            assert ht2 == ht and n == nb and n >= ht * wv, info
        # the MMA's N: a multiple of 16 within the accumulator buffer
        assert n % 16 == 0 and 32 <= n <= (240 if code == bt.BT_CODE_E2M1 else 256), info
        # the staged rows hold every tap's shifted view of a CTA's columns
        assert rv * wv >= nb + info["max_tap_shift"], info
        assert 1 <= info["phases"] <= s * s
        assert info["pixel_stages"] in (1, 2) and info["smem_bytes"] <= 227 * 1024
        # tiles: channel tiles x images x bands
        per = 256 if info["pair"] else 128
        assert info["tiles"] == -(-O // per) * B * bands
        # a split never gives fewer bands than the planner's
        if split > 1:
            base = bt.bt_conv2d_plan_info(B, C, H, W, O, k, s, p, d, code, od, 152, info["pair"], 1)
            assert bands >= base["bands"]
    assert seen > 0


def test_plan_info_rejects_bad_arguments():
    ok = (2, 64, 14, 14, 64, 3, 1, 1, 1)
    with pytest.raises(bt.BtError):
        bt.bt_conv2d_plan_info(*ok, bt.BT_CODE_BITS)
    with pytest.raises(bt.BtError):
        bt.bt_conv2d_plan_info(*ok, bt.BT_CODE_E2M1, sms=0)
    with pytest.raises(bt.BtError):
        bt.bt_conv2d_plan_info(*ok, bt.BT_CODE_E2M1, pair=2)
    with pytest.raises(bt.BtError):
        bt.bt_conv2d_plan_info(*ok, bt.BT_CODE_E2M1, split=0)
    with pytest.raises(bt.BtError):
        bt.bt_conv2d_plan_info(2, 64, 2, 2, 64, 5, 1, 0, 1, bt.BT_CODE_E2M1)      # no output pixel


def test_explicit_route_reports_no_implicit_plan(monkeypatch):
    monkeypatch.setenv("BT_CONV_IMPLICIT", "0")
    assert bt.bt_conv2d_plan_info(2, 64, 14, 14, 64, 3, 1, 1, 1, bt.BT_CODE_E2M1)["implicit"] == 0
