"""GPU parity of dsa_index_store: stored bytes must equal the oracle's bit for bit."""
import numpy as np
import pytest

from oracle import store as S
from synth import inputs as I
from tests import gpu_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import torch
    from dsa_sparse_attention_store_gb300 import Context
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    c = Context(theta=10000.0, eps=1e-6, max_pos=131072)
    yield c
    c.close()


def _compare_cache(wl, fmt, d, pos, seq):
    got = d["cache"].cpu().numpy()
    want = S.new_cache(wl.num_pages, fmt)
    S.store(want, fmt, wl.new_k, wl.new_pos, wl.new_seq, wl.page_table, wl.num_pages, wl.theta, wl.eps)
    gb = U.slot_bytes(got, fmt, wl, pos, seq)
    wb = U.slot_bytes(want, fmt, wl, pos, seq)
    bad = np.nonzero(np.any(gb != wb, axis=1))[0]
    assert len(bad) == 0, f"{len(bad)} tokens differ, first at token {bad[0]}"


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
def test_store_bitexact_small(ctx, fmt):
    wl = I.make_workload("st", [300, 777, 129, 64, 1], [1] * 5, [300, 777, 129, 64, 1], True, 512,
                         seed=21, wid=20)
    d = U.device_workload(wl, fmt, ctx, store_fill=False)
    assert ctx.device_status() == 0
    _compare_cache(wl, fmt, d, wl.new_pos, wl.new_seq)
    # untouched slots stay zero (last page of sequence 0 holds 300 % 64 = 44 tokens)
    got = d["cache"].cpu().numpy()
    page = int(wl.page_table[0, 4])
    pb = S.PAGE_BYTES[fmt]
    tb = 256 if fmt == S.FMT_BF16 else S.CODE_BYTES[fmt]
    assert np.all(got[page * pb + 44 * tb: page * pb + 64 * tb] == 0)


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
def test_store_bitexact_extreme_values(ctx, fmt):
    # wide dynamic range, zero rows, tiny rows, rows with one huge element
    rng = np.random.default_rng(5)
    T = 512
    x = rng.standard_normal((T, 128)) * np.exp(rng.uniform(-20, 20, (T, 1)))
    x[0] = 0.0
    x[1] = 1e-38
    x[2, :] = 1e-3
    x[2, 17] = 3e4
    x[3] = rng.standard_normal(128) * np.exp(rng.uniform(-30, 30, 128))
    wl = I.make_workload("ex", [T], [1], [T], True, 512, seed=22, wid=21)
    wl.new_k = I.to_bf16_bits(x.astype(np.float32))
    d = U.device_workload(wl, fmt, ctx, store_fill=False)
    assert ctx.device_status() == 0
    _compare_cache(wl, fmt, d, wl.new_pos, wl.new_seq)


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
def test_store_bitexact_tiny_prefill(ctx, fmt):
    wl = I.tiny_prefill()
    d = U.device_workload(wl, fmt, ctx, store_fill=False)
    _compare_cache(wl, fmt, d, wl.new_pos, wl.new_seq)


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
def test_store_bitexact_long_positions(ctx, fmt):
    # the long-decode append: 8 sequences x 256 tokens at positions 130816..131071
    wl = I.make_workload("ap", [131072] * 8, [1] * 8, [256] * 8, True, 1024, seed=0, wid=4)
    d = U.device_workload(wl, fmt, ctx, store_fill=False)
    assert ctx.device_status() == 0
    _compare_cache(wl, fmt, d, wl.new_pos, wl.new_seq)


def test_store_rejects_bad_page_on_device(ctx):
    import torch
    wl = I.make_workload("bp", [128], [1], [128], True, 512, seed=23, wid=22)
    wl.page_table[0, 1] = wl.num_pages + 5   # positions 64..127 point past the cache
    d = U.device_workload(wl, 0, ctx, store_fill=False, store_new=False)
    k = U.t_bf16(wl.new_k).cuda()
    pos = torch.from_numpy(wl.new_pos).cuda()
    seq = torch.from_numpy(wl.new_seq).cuda()
    ctx.store(k, pos, seq, d["page_table"], d["cache"], wl.num_pages, 0)
    assert ctx.device_status() == 4          # DSA_ERR_DEVICE_BOUNDS, no trap
    assert ctx.device_status() == 0          # the word was cleared
    # the valid half was still stored correctly
    got = d["cache"].cpu().numpy()
    want = S.new_cache(wl.num_pages, 0)
    S.store(want, 0, wl.new_k[:64], wl.new_pos[:64], wl.new_seq[:64], wl.page_table, wl.num_pages)
    assert np.array_equal(U.slot_bytes(got, 0, wl, wl.new_pos[:64], wl.new_seq[:64]),
                          U.slot_bytes(want, 0, wl, wl.new_pos[:64], wl.new_seq[:64]))


def _pipeline_tokens():
    # several waves of store CTAs (8 tokens each) and a ragged tail: 3 x 64
    # tokens per SM plus 37 (the last 8-token chunk holds five tokens on a
    # 152-SM part, and one warp of its CTA straddles the end of the batch;
    # with 3 sequences the CTAs visit the chunks in 3 interleaved regions,
    # and the last region has one chunk past the end)
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 3 * 16 * 4 * sms + 37


@pytest.mark.parametrize("fmt", [S.FMT_BF16, S.FMT_FP8, S.FMT_FP4])
def test_store_bitexact_several_waves(ctx, fmt):
    T = _pipeline_tokens()
    lens = [T // 3 + 5, T // 3 - 11, T - 2 * (T // 3) + 6]
    wl = I.make_workload("pl", lens, [1] * 3, lens, True, 512, seed=24, wid=23)
    assert wl.new_pos.shape[0] == T
    d = U.device_workload(wl, fmt, ctx, store_fill=False)
    assert ctx.device_status() == 0
    _compare_cache(wl, fmt, d, wl.new_pos, wl.new_seq)


def test_store_bad_pages_inside_a_long_run(ctx):
    # two pages in the middle of a multi-token run point past the cache: those
    # 128 tokens are dropped and reported, every other token is stored exactly
    import torch
    T = _pipeline_tokens()
    wl = I.make_workload("pb", [T], [1], [T], True, 512, seed=25, wid=24)
    bad_pages = [7, wl.page_table.shape[1] // 2]
    for pg in bad_pages:
        wl.page_table[0, pg] = wl.num_pages + pg
    d = U.device_workload(wl, 0, ctx, store_fill=False, store_new=False)
    k = U.t_bf16(wl.new_k).cuda()
    pos = torch.from_numpy(wl.new_pos).cuda()
    seq = torch.from_numpy(wl.new_seq).cuda()
    ctx.store(k, pos, seq, d["page_table"], d["cache"], wl.num_pages, 0)
    assert ctx.device_status() == 4          # DSA_ERR_DEVICE_BOUNDS
    assert ctx.device_status() == 0
    keep = ~np.isin(wl.new_pos // 64, bad_pages)
    assert keep.sum() == T - 128
    got = d["cache"].cpu().numpy()
    want = S.new_cache(wl.num_pages, 0)
    S.store(want, 0, wl.new_k[keep], wl.new_pos[keep], wl.new_seq[keep], wl.page_table, wl.num_pages)
    assert np.array_equal(U.slot_bytes(got, 0, wl, wl.new_pos[keep], wl.new_seq[keep]),
                          U.slot_bytes(want, 0, wl, wl.new_pos[keep], wl.new_seq[keep]))
