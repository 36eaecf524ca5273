"""Host logic without a GPU: the seeded mask generators' structure, and the
benchmark's counts (tiles a pass runs under a mask's live spans, the D_i
kernel's algorithmic bytes), pinned on cases whose answers are known by hand."""
import math

import torch

import bench
from attention_backward_tcgen05_gb300 import inputs

NEG = float("-inf")


def _live(mask):
    return mask.float() != NEG


def test_operands_do_not_depend_on_the_mask_kind():
    # q, k, v and d are drawn before the mask, so every mask kind sees the
    # same operands for one seed and shape
    base = inputs.make(inputs.custom(1, 2, 1, 70, 90, 16, mask="none", seed=5))
    for kind in ("random", "pad", "docs", "band"):
        x = inputs.make(inputs.custom(1, 2, 1, 70, 90, 16, mask=kind, seed=5))
        for key in ("q", "k", "v", "d"):
            assert torch.equal(x[key], base[key]), (kind, key)
        assert x["mask"].dtype == torch.float16 and x["mask"].shape == (70, 90)


def test_docs_mask_is_block_diagonal():
    # with no Bernoulli part, query n and key m are live together exactly
    # when they fall in the same document: the live set is a union of
    # rectangles along the diagonal, and the document of n (of m) never
    # decreases as n (m) grows
    w = inputs.custom(1, 1, 1, 300, 500, 8, mask="docs", mask_p=0.0, parts=4, seed=9)
    live = _live(inputs.make(w)["mask"])
    first = [int(torch.nonzero(live[n]).min()) for n in range(300)]
    last = [int(torch.nonzero(live[n]).max()) for n in range(300)]
    assert first == sorted(first) and last == sorted(last)
    for n in range(300):
        # each row's live keys are one contiguous run
        assert int(live[n].sum()) == last[n] - first[n] + 1
    # rows of one document share the run; the runs of two documents are disjoint
    runs = sorted(set(zip(first, last)))
    assert 1 <= len(runs) <= 4
    for (a0, a1), (b0, b1) in zip(runs, runs[1:]):
        assert a1 < b0
    assert runs[0][0] == 0 and runs[-1][1] == 499


def test_band_mask_keeps_keys_near_the_scaled_diagonal():
    w = inputs.custom(1, 1, 1, 200, 400, 8, mask="band", mask_p=0.0, parts=1, seed=3)
    live = _live(inputs.make(w)["mask"])
    n = torch.arange(200, dtype=torch.float64)[:, None]
    m = torch.arange(400, dtype=torch.float64)[None, :]
    assert torch.equal(live, (m - n * 400 / 200).abs() <= 128)


def test_pad_mask_padding_rows_and_columns():
    w = inputs.custom(1, 1, 1, 160, 240, 8, mask="pad", mask_p=0.0, seed=4)
    live = _live(inputs.make(w)["mask"])
    mv, nv = 240 * 5 // 8 + 3, 160 * 7 // 8 + 1
    want = torch.zeros((160, 240), dtype=torch.bool)
    want[:nv, :mv] = True
    assert torch.equal(live, want)


def test_bernoulli_part_rate():
    w = inputs.custom(1, 1, 1, 256, 512, 8, mask="docs", mask_p=0.25, parts=1, seed=12)
    live = _live(inputs.make(w)["mask"])  # one document: only the Bernoulli part masks
    rate = 1.0 - live.double().mean().item()
    assert abs(rate - 0.25) < 4 * math.sqrt(0.25 * 0.75 / live.numel())


def _block_mask(N, M, blocks):
    """f16 mask with -inf everywhere but the listed (query rows, key rows) blocks."""
    mask = torch.full((N, M), NEG)
    for (n0, n1), (m0, m1) in blocks:
        mask[n0:n1, m0:m1] = 0.0
    return mask.to(torch.float16)


def test_tiles_run_two_tile_aligned_documents():
    # 4 x 4 tiles, two documents of 2 x 2 tiles on the diagonal: each tile
    # row's live span is 2 tiles of 4, for both passes
    w = inputs.custom(1, 1, 1, 512, 512, 8, mask="docs")
    mask = _block_mask(512, 512, [((0, 256), (0, 256)), ((256, 512), (256, 512))])
    assert bench.executed_tile_fraction(w, mask, 3) == 0.5
    assert bench.executed_tile_fraction(w, mask, 4) == 0.5
    assert bench.executed_tile_fraction(w, None, 3) == 1.0


def test_tiles_run_span_includes_interior_dead_tiles_and_empty_rows():
    # query tile 0 has live tiles 0 and 3 (span 4 tiles, the two between
    # still run); query tile 1 has none (the query pass still runs one tile);
    # query tiles 2, 3 live in key tile 1 only
    w = inputs.custom(1, 1, 1, 512, 512, 8, mask="docs")
    mask = _block_mask(512, 512, [((0, 1), (0, 1)), ((5, 6), (400, 401)), ((256, 512), (128, 256))])
    # query pass: 4 + 1 + 1 + 1 of 16 tiles
    assert bench.executed_tile_fraction(w, mask, 3) == 7 / 16
    # key pass: key tile 0 -> query tiles 0..0, key tile 1 -> 2..3, key tile 2
    # -> none, key tile 3 -> 0..0: 1 + 2 + 0 + 1 of 16
    assert bench.executed_tile_fraction(w, mask, 4) == 4 / 16


def test_tiles_run_with_causal_bound():
    # causal (top-left), 3 x 3 tiles, mask live everywhere but key tile 0:
    # query pass rows run key tiles 1..min(qt, 2) -> 0 live in row 0 (one
    # tile run), 1, 2 of 1 + 2 + 3 causal tiles; key pass columns 1 and 2 run
    # query tiles 1..2 and 2..2, column 0 none, of 3 + 2 + 1
    w = inputs.custom(1, 1, 1, 384, 384, 8, mask="docs", causal=True)
    mask = _block_mask(384, 384, [((0, 384), (128, 384))])
    assert bench.executed_tile_fraction(w, mask, 3) == (1 + 1 + 2) / (1 + 2 + 3)
    assert bench.executed_tile_fraction(w, mask, 4) == (0 + 2 + 1) / (3 + 2 + 1)


def test_preprocess_bytes():
    # dO and O read (bf16), D_i written (f32), padding zeroed: DK = 5 gives
    # 1 padding float after dQ (B*H*N*5 = 30 floats -> 32), K and V slices
    # B*Hkv*M*5 = 35 floats -> 36 each
    w = inputs.custom(1, 2, 1, 3, 7, 5, 5, dtype="bf16")
    rows = 1 * 2 * 3
    assert bench.preprocess_bytes(w) == 2 * rows * 5 * 2 + rows * 4 + (2 + 1 + 1) * 4
    g = inputs.WORKLOADS["gqa_causal_d128"]
    assert bench.preprocess_bytes(g) == 2 * 4 * 32 * 2048 * 128 * 2 + 4 * 32 * 2048 * 4
