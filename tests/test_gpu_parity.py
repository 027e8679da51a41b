"""GPU path vs the CPU oracle, element by element, through the C ABI (needs a GB300).

Every comparison is bit-exact: each output row, taken as a set of int32 slots,
must equal the oracle's, and the un-mapped selection must pass the complete
invariant check of tests/checks.py. Inputs come from workloads.py (seeded, on
the host) and are copied to the device unchanged.
"""

from __future__ import annotations

import contextlib

import numpy as np
import pytest

import oracle
import workloads
from checks import check_workload, same_sets

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_attention_indexer_sm_gb300 as p
    p.load_library()
    return p


@pytest.fixture(autouse=True)
def no_guard_hits(pkg):
    """No internal consistency check of the kernels fails in any test."""
    pkg.topk_reset_guard_hits()
    yield
    assert pkg.topk_guard_hits() == 0, "a kernel's internal consistency check failed"


@contextlib.contextmanager
def settings(pkg, split=None, tie_cap=None, fast=None, cta=None, staged=None, chip=None):
    if split is not None and chip is None:
        chip = 0  # a forced cluster split is what such a test exercises
    prev_chip = pkg.topk_set_chip_split(chip) if chip is not None else None
    prev_split = pkg.topk_set_row_split(split) if split is not None else None
    prev_cap = pkg.topk_set_tie_capacity(tie_cap) if tie_cap is not None else None
    prev_fast = pkg.topk_set_fast_tier(fast) if fast is not None else None
    prev_cta = pkg.topk_set_cta_threads(cta) if cta is not None else None
    prev_staged = pkg.topk_set_staged_tier(staged) if staged is not None else None
    try:
        yield
    finally:
        if chip is not None:
            pkg.topk_set_chip_split(prev_chip)
        if staged is not None:
            pkg.topk_set_staged_tier(prev_staged)
        if cta is not None:
            pkg.topk_set_cta_threads(prev_cta)
        if split is not None:
            pkg.topk_set_row_split(prev_split)
        if tie_cap is not None:
            pkg.topk_set_tie_capacity(prev_cap)
        if fast is not None:
            pkg.topk_set_fast_tier(prev_fast)


def run_gpu(pkg, w, stream=None) -> np.ndarray:
    dev = torch.device("cuda:0")
    scores = torch.from_numpy(np.ascontiguousarray(w.scores)).to(dev)
    seq = torch.from_numpy(np.ascontiguousarray(w.seq_lens)).to(dev)
    out = torch.full((w.batch, w.k), -7, dtype=torch.int32, device=dev)  # poison
    if w.form == "raw":
        pkg.topk_transform_raw(scores, seq, w.k, out=out, stream=stream)
    elif w.form == "paged":
        pt = torch.from_numpy(np.ascontiguousarray(w.page_table)).to(dev)
        pkg.topk_transform_paged(scores, seq, pt, w.page_size, w.k, out=out, stream=stream)
    elif w.form == "window":
        st = torch.from_numpy(np.ascontiguousarray(w.row_starts)).to(dev)
        # the window-length hint on the prefill workloads, none (the row length) on the rest
        hint = w.max_row_len if w.name.startswith("window_b") else 0
        pkg.topk_transform_window(scores, st, seq, w.k, max_row_len_hint=hint, out=out,
                                  stream=stream)
    else:
        rs = torch.from_numpy(np.ascontiguousarray(w.row_starts)).to(dev)
        hint = int(np.max(w.seq_lens, initial=0))
        pkg.topk_transform_ragged(scores, rs, seq, w.k, max_row_len_hint=hint, out=out,
                                  stream=stream)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def assert_parity(w, got, check_rows=None):
    exp = oracle.run(w)
    ok = same_sets(got, exp)
    if not ok.all():
        b = int(np.flatnonzero(~ok)[0])
        diff = np.setxor1d(got[b], exp[b])
        raise AssertionError(f"{w.name}: {int((~ok).sum())} rows differ from the oracle; "
                             f"row {b} symmetric difference {diff[:10].tolist()}")
    errs = check_workload(w, got, max_rows=check_rows)
    assert not errs, f"{w.name}: {errs[:3]}"


# ------------------------------------------------------------ the pages' workloads

def test_config1_unit_shape(pkg):
    w = workloads.config1()
    assert_parity(w, run_gpu(pkg, w))


@pytest.mark.parametrize("bs", [1, 48])
@pytest.mark.parametrize("c4_len", [2048, 8192, 32768])
def test_unit_test_shapes(pkg, bs, c4_len):
    """The parameter grid of test_deepseek_v4_topk_transform (PR #36004 page)."""
    w = workloads.unit_test_shape(bs, c4_len)
    assert_parity(w, run_gpu(pkg, w))


@pytest.mark.parametrize("c4_len", [8192, 32768])
def test_config2_random_lengths(pkg, c4_len):
    w = workloads.config2(c4_len)
    assert_parity(w, run_gpu(pkg, w))


@pytest.mark.parametrize("form", ["raw", "paged"])
@pytest.mark.parametrize("batch", [1, 8, 64, 128, 256])
def test_config3_decode_sweep(pkg, batch, form):
    w = workloads.config3(batch, form)
    assert_parity(w, run_gpu(pkg, w), check_rows=16)


@pytest.mark.parametrize("dist", ["banded", "narrow", "subnormal"])
def test_config4_adversarial_ragged(pkg, dist):
    w = workloads.config4(dist)
    assert_parity(w, run_gpu(pkg, w), check_rows=4)


@pytest.mark.parametrize("batch", [1, 2, 4])
def test_config5_long_rows(pkg, batch):
    """Small batches of 262144-element rows: the chip-wide split from 4 rows on
    (automatic), clusters below."""
    assert (pkg.topk_workspace_bytes(batch, 262144, 2048) > 0) == (batch >= 4)
    w = workloads.config5(batch)
    assert_parity(w, run_gpu(pkg, w), check_rows=2)


@pytest.mark.parametrize("batch,chip", [(1, 2), (4, 0)])
def test_config5_long_rows_other_path(pkg, batch, chip):
    """The same rows on the path the automatic rule does not pick: the chip-wide split
    for one row, clusters for four."""
    w = workloads.config5(batch)
    with settings(pkg, chip=chip):
        assert (pkg.topk_workspace_bytes(batch, 262144, 2048) > 0) == (chip == 2)
        got = run_gpu(pkg, w)
    assert_parity(w, got, check_rows=2)


# ------------------------------------------------------------ the chip-wide split

@pytest.mark.parametrize("tie_cap", [None, 0, 16, 300])
@pytest.mark.parametrize("dist", ["normal", "decode", "banded", "narrow", "subnormal", "heavy_tail"])
def test_chip_split_forced(pkg, dist, tie_cap):
    """The chip-wide split forced onto paged rows of random lengths (some shorter than
    k); small tie capacities shrink its candidate stores, so rows take its fallback."""
    w = _mixed(900, dist)
    with settings(pkg, chip=2, tie_cap=tie_cap):
        assert pkg.topk_workspace_bytes(w.batch, w.scores.shape[1], w.k) > 0
        got = run_gpu(pkg, w)
    assert_parity(w, got)


@pytest.mark.parametrize("k", [1, 7, 1024, 2048])
@pytest.mark.parametrize("form", ["raw", "ragged", "window"])
def test_chip_split_forms(pkg, form, k):
    """Every form through the chip-wide split: odd row offsets, empty rows, rows
    shorter than k, duplicates."""
    g = workloads.rng(910 + k)
    if form == "ragged":
        lens = np.array([0, 1, 2047, 2048, 2049, 70001, 3, 150000, 0, 65536], np.int64)
        gaps = g.integers(0, 7, size=lens.shape[0])
        starts = (np.concatenate([[0], np.cumsum(lens + gaps)[:-1]]) + 1).astype(np.int32)
        total = int(starts[-1] + lens[-1] + 5)
        scores = workloads.row_values(g, "banded", total, dup=True)
        w = workloads.Workload(f"chip_ragged_k{k}", "ragged", k, scores, lens.astype(np.int32),
                               None, 64, starts)
    elif form == "window":
        batch, stride = 5, 70001
        scores = workloads.random_rows(g, batch, stride, "decode", dup=True)
        hi = g.integers(0, stride + 3, size=batch).astype(np.int32)
        lo = (hi * g.random(batch) * 0.5).astype(np.int32)
        w = workloads.Workload(f"chip_window_k{k}", "window", k, scores, hi, None, 64, lo)
    else:
        w = _mixed(920 + k, "heavy_tail", batch=5, stride=70001, k=k).as_raw()
    with settings(pkg, chip=2):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


@pytest.mark.parametrize("dist", ["banded", "narrow", "subnormal"])
def test_chip_split_exact_tier_on_clusters(pkg, dist):
    """Long concentrated rows through the chip-wide split (automatic for 4 rows): their
    candidates overflow the per-CTA stores, so the select kernel's cluster runs the exact
    tier over each row."""
    w = _mixed(940, dist, batch=4, stride=100003, k=2048)
    assert pkg.topk_workspace_bytes(w.batch, w.scores.shape[1], w.k) > 0
    assert_parity(w, run_gpu(pkg, w), check_rows=2)


def test_chip_split_workspace(pkg):
    """A caller's workspace, reused without initialisation, gives the same rows; one
    too small sends the call to the cluster path, with the same result."""
    w = workloads.config5(4)
    dev = torch.device("cuda:0")
    scores = torch.from_numpy(w.scores).to(dev)
    seq = torch.from_numpy(w.seq_lens).to(dev)
    pt = torch.from_numpy(w.page_table).to(dev)
    need = pkg.topk_workspace_bytes(w.batch, w.scores.shape[1], w.k)
    assert need > 0
    ws = torch.full((need,), 0xA5, dtype=torch.uint8, device=dev)  # garbage contents
    outs = []
    for wsx in (ws, ws, ws[: need - 256]):
        out = torch.full((w.batch, w.k), -7, dtype=torch.int32, device=dev)
        pkg.topk_transform_paged(scores, seq, pt, w.page_size, w.k, out=out, workspace=wsx)
        outs.append(out.cpu().numpy())
    torch.cuda.synchronize()
    for got in outs:
        assert_parity(w, got, check_rows=1)


# ------------------------------------------------------------ a page table narrower than a row

@pytest.mark.parametrize("split,fast", [(None, 1), (None, 0), (4, 1), (4, 0)])
def test_paged_table_narrower_than_row(pkg, split, fast):
    """Rows that need more pages than the table's row stride holds: the kernel reads
    only the row's own entries, writes -1 for each selected position whose page is
    missing, and counts each such row once in the guard counter (called through the C
    ABI directly: the binding refuses such a table)."""
    import ctypes
    lib = pkg.load_library()
    g = workloads.rng(4242)
    B, S, ps, npt, k = 4, 8192, 64, 100, 1024
    scores = workloads.random_rows(g, B, S, "normal")
    seq = np.array([8192, 6400, 6000, 8000], np.int32)   # rows 0 and 3 need 128 and 125 pages
    table = np.stack([g.permutation(4 * npt)[:npt] for _ in range(B)]).astype(np.int32)
    raw = oracle.run(workloads.Workload("narrow_table_raw", "raw", k, scores, seq, None, ps))
    page = np.where(raw >= 0, raw // ps, 0)
    exp = np.where((raw >= 0) & (page < npt),
                   np.take_along_axis(table, np.minimum(page, npt - 1), 1) * ps + raw % ps, -1)
    dev = torch.device("cuda:0")
    d_scores = torch.from_numpy(scores).to(dev)
    d_seq = torch.from_numpy(seq).to(dev)
    d_pt = torch.from_numpy(table).to(dev)
    d_out = torch.full((B, k), -7, dtype=torch.int32, device=dev)
    with settings(pkg, split=split, fast=fast):
        st = lib.topk_transform_paged(ctypes.c_void_p(d_scores.data_ptr()), S,
                                      ctypes.c_void_p(d_seq.data_ptr()),
                                      ctypes.c_void_p(d_pt.data_ptr()), npt, ps, B, k,
                                      ctypes.c_void_p(d_out.data_ptr()), None, 0, None)
        torch.cuda.synchronize()
    assert st == 0
    got = d_out.cpu().numpy()
    assert same_sets(got, exp).all()
    assert pkg.topk_guard_hits() == 2  # one per row that needs more pages than the stride
    pkg.topk_reset_guard_hits()


# ------------------------------------------------------------ every execution path

def _mixed(seed, dist, batch=6, stride=20000, k=1024, dup=True, form="paged"):
    g = workloads.rng(seed)
    scores = workloads.random_rows(g, batch, stride, dist, dup)
    seq = g.integers(k // 2, stride + 5, size=batch).astype(np.int32)
    pt = workloads.permuted_page_table(g, batch, workloads.pages_for(stride, 64))
    w = workloads.Workload(f"{dist}_{form}_s{seed}", form, k, scores, seq, pt, 64)
    return w


@pytest.mark.parametrize("fast", [True, False])
@pytest.mark.parametrize("split", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("dist", ["normal", "decode", "banded", "narrow", "subnormal", "heavy_tail"])
def test_every_row_split(pkg, split, dist, fast):
    """Single-CTA and cluster row-split paths, with and without the sampled filter
    tier, give the oracle's set (cross-path A/B of the PR #36004 page's index-set
    comparison, restated per path)."""
    w = _mixed(100 + split, dist)
    with settings(pkg, split=split, fast=fast):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


@pytest.mark.parametrize("fast", [True, False])
@pytest.mark.parametrize("tie_cap", [0, 1, 16, 300, 4096])
@pytest.mark.parametrize("split", [1, 4])
@pytest.mark.parametrize("dist", ["decode", "banded", "narrow", "subnormal"])
def test_tie_buffer_capacity(pkg, tie_cap, split, dist, fast):
    """Small buffers force the filter's overflow fallback, more radix rounds and the
    position-ordered rescan."""
    w = _mixed(200 + tie_cap, dist, k=2048)
    with settings(pkg, split=split, tie_cap=tie_cap, fast=fast):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


@pytest.mark.parametrize("staged", [2, 3, 0])
@pytest.mark.parametrize("tie_cap", [0, 16, 300, 4096])
@pytest.mark.parametrize("dist", ["normal", "decode", "banded", "narrow", "subnormal", "heavy_tail"])
def test_single_cta_tiers(pkg, dist, tie_cap, staged):
    """Rows owned by one CTA on the staged tier (the row copied to shared memory from
    kernel start, whole or by halves) and on the streaming fast tier, with every
    buffer size down to none (the exact-tier fallback inside each)."""
    w = _mixed(900 + tie_cap, dist, k=1024 if tie_cap != 300 else 2048)
    with settings(pkg, split=1, tie_cap=tie_cap, staged=staged):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


@pytest.mark.parametrize("staged", [2, 3, 0])
@pytest.mark.parametrize("form", ["raw", "paged"])
@pytest.mark.parametrize("batch", [64, 256])
def test_decode_sweep_both_single_cta_tiers(pkg, batch, form, staged):
    """The decode sweep on both single-CTA tiers (the streaming tier reads candidates
    back from L2 below one row per SM and from L1 above)."""
    w = workloads.config3(batch, form)
    with settings(pkg, staged=staged):
        got = run_gpu(pkg, w)
    assert_parity(w, got, check_rows=8)


@pytest.mark.parametrize("staged", [2, 3])
@pytest.mark.parametrize("stride", [1, 3, 4, 5, 127, 1025, 4097, 8191, 30001, 32764, 32767, 32768])
def test_staged_tier_strides(pkg, stride, staged):
    """Row strides of every alignment up to the staged tier's limit, with lengths from
    zero to the stride (unaligned heads and tails, partial runs and bands)."""
    g = workloads.rng(1300 + stride)
    batch, k = 9, 700
    scores = workloads.random_rows(g, batch, stride, "decode", dup=True)
    seq = np.array([stride, stride - 1, stride // 2, k, k + 1, 4097, 0, -5, 1], np.int32)
    seq = np.minimum(seq, stride)
    pt = workloads.permuted_page_table(g, batch, workloads.pages_for(stride, 16))
    for form in ("raw", "paged"):
        w = workloads.Workload(f"staged_stride{stride}_{form}", form, k, scores, seq,
                               pt if form == "paged" else None, 16)
        with settings(pkg, staged=staged):
            got = run_gpu(pkg, w)
        assert_parity(w, got)


@pytest.mark.parametrize("staged", [2, 3])
def test_staged_tier_short_hint_falls_back(pkg, staged):
    """Ragged rows longer than their length hint promised: the staged tier cannot hold
    them and runs the exact tier instead."""
    g = workloads.rng(1400)
    lens = np.array([40000, 33000, 32768, 12000, 0, 70000], np.int32)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int32) + 3
    flat = workloads.random_rows(g, 1, int(starts[-1] + lens[-1] + 5), "decode")[0]
    w = workloads.Workload("ragged_short_hint", "ragged", 1024, flat, lens, None, 64,
                           row_starts=starts)
    dev = torch.device("cuda:0")
    out = torch.full((w.batch, w.k), -7, dtype=torch.int32, device=dev)
    with settings(pkg, staged=staged):
        pkg.topk_transform_ragged(torch.from_numpy(flat).to(dev), torch.from_numpy(starts).to(dev),
                                  torch.from_numpy(lens).to(dev), w.k, max_row_len_hint=20000,
                                  out=out)
        torch.cuda.synchronize()
    assert_parity(w, out.cpu().numpy())


@pytest.mark.parametrize("staged", [2, 3])
def test_staged_tier_forms(pkg, staged):
    """Ragged and window rows on the staged tier (their data start comes with the
    length), including windows that start and end anywhere in the row."""
    g = workloads.rng(1500 + staged)
    lens = np.array([30000, 5000, 32768, 1024, 0, 9000, 17], np.int32)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int32) + 1
    flat = workloads.random_rows(g, 1, int(starts[-1] + lens[-1] + 3), "decode", dup=True)[0]
    rag = workloads.Workload("staged_ragged", "ragged", 1000, flat, lens, None, 64, row_starts=starts)
    win = workloads.prefill_windows(40, 32768, window=20000, k=1000)
    with settings(pkg, staged=staged):
        got_r = run_gpu(pkg, rag)
        got_w = run_gpu(pkg, win)
    assert_parity(rag, got_r)
    assert_parity(win, got_w)


@pytest.mark.parametrize("split", [1, 2, 8])
def test_misleading_sample_falls_back(pkg, split):
    """Large values placed exactly on the sampled quads make the sampled threshold
    too high (fewer than k candidates); the verify step must send the row to the
    exact tier. Every 16-byte quad position is made large in turn for one row, so
    whatever the sample stride, some rows are misled."""
    batch, stride, k = 16, 32768, 1024
    g = workloads.rng(800 + split)
    scores = workloads.random_rows(g, batch, stride, "normal")
    for b in range(batch):
        period = 2 ** (b % 8 + 1)  # quad strides 2 .. 256
        quads = np.arange(0, stride // 4, period)
        for c in range(4):
            scores[b, quads * 4 + c] = 100.0 + g.standard_normal(quads.shape[0]).astype(np.float32)
    seq = np.full(batch, stride, np.int32)
    w = workloads.Workload("misleading_sample", "raw", k, scores, seq)
    with settings(pkg, split=split):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


@pytest.mark.parametrize("tie_cap", [None, 300])
@pytest.mark.parametrize("split", [2, 8, 16, "chip"])
def test_misleading_sample_window_falls_back(pkg, split, tie_cap):
    """Rows packed into a few values send a cluster row (and a chip-wide split row whose
    candidates overflow) to the exact tier, whose first round looks only at the sample's
    window of keys. Here the sample is wrong on purpose, and the rounds must start again
    from the top bits. Each CTA of a cluster samples runs of 32 quads at a power-of-two
    spacing of at least 256 quads (for these rows and splits; 1024 in the chip-wide
    split's filter), so quads at offsets 32 .. 63 of every 64 are never sampled.
    Row 0: constant 5.0 with 65536 larger values off the sample (the k-th key is above
    the window). Row 1: the same with 8192 larger values. Row 2: 1024 larger values,
    all on the sample (the window is above the k-th key). Row 3: a 'narrow' row, whose
    window is right."""
    batch, stride, k = 4, 262144, 2048
    g = workloads.rng(900 + (split if split != "chip" else 1))
    scores = np.full((batch, stride), 5.0, np.float32)
    q = np.arange(stride // 4)
    off_sample = [q[(q % 64 >= 32) & (q % 64 < 48)], q[(q % 256 >= 32) & (q % 256 < 40)]]
    for b, quads in enumerate(off_sample):
        for c in range(4):
            scores[b, quads * 4 + c] = 6.0 + 1e-3 * g.standard_normal(quads.shape[0]).astype(np.float32)
    on_sample = q[(q % 512 == 0) | (q % 512 == 16)]
    for c in range(4):
        scores[2, on_sample * 4 + c] = 6.0 + 1e-3 * g.standard_normal(on_sample.shape[0]).astype(np.float32)
    scores[3] = workloads.random_rows(g, 1, stride, "narrow")[0]
    seq = np.full(batch, stride, np.int32)
    w = workloads.Workload("misleading_sample_window", "raw", k, scores, seq)
    with (settings(pkg, chip=2, tie_cap=tie_cap) if split == "chip"
          else settings(pkg, split=split, tie_cap=tie_cap)):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


@pytest.mark.parametrize("cta,tie_cap", [(None, None), (None, 300), (256, None)])
@pytest.mark.parametrize("batch", [8, 160])
def test_single_cta_overflow_window(pkg, batch, cta, tie_cap):
    """Single-CTA rows whose filter overflows start the exact tier from the bits that the
    ends of the candidate bins' span share; here that window is wrong on purpose in half
    the rows. A single CTA samples runs of 32 quads at a spacing of 512 quads (32768
    elements, either build), so quads at offsets 32 .. 47 of every 64 are never sampled.
    Rows 0 and 1: N(0, 1) and constant 5.0, each with 8192 values near 6.0 off the sample
    (the k-th key is above the window). Rows 2 and 3: 'banded' and 'narrow' rows. 160 rows
    take the filter that reads candidate values back from L1."""
    stride, k = 32768, 1024
    g = workloads.rng(960 + batch)
    base = np.stack([g.standard_normal(stride).astype(np.float32),
                     np.full(stride, 5.0, np.float32),
                     workloads.random_rows(g, 1, stride, "banded")[0],
                     workloads.random_rows(g, 1, stride, "narrow")[0]])
    q = np.arange(stride // 4)
    off = q[(q % 64 >= 32) & (q % 64 < 48)]
    for b in range(2):
        for c in range(4):
            base[b, off * 4 + c] = 6.0 + 1e-3 * g.standard_normal(off.shape[0]).astype(np.float32)
    scores = np.ascontiguousarray(np.tile(base, (batch // 4, 1)))
    seq = np.full(batch, stride, np.int32)
    w = workloads.Workload("single_cta_overflow_window", "raw", k, scores, seq)
    with settings(pkg, split=1, staged=0, cta=cta, tie_cap=tie_cap):
        got = run_gpu(pkg, w)
    assert_parity(w, got, check_rows=8)


@pytest.mark.parametrize("form", ["raw", "paged"])
@pytest.mark.parametrize("batch", [1, 64, 256])
def test_exact_tier_alone_on_decode_sweep(pkg, batch, form):
    w = workloads.config3(batch, form)
    with settings(pkg, fast=False):
        got = run_gpu(pkg, w)
    assert_parity(w, got, check_rows=8)


@pytest.mark.parametrize("split", [1, 2, 16])
def test_all_equal_rows(pkg, split):
    """Every key ties: the first k positions win."""
    batch, stride, k = 3, 50000, 2048
    scores = np.full((batch, stride), 1.5, np.float32)
    scores[1, ::7] = -0.0
    scores[2] = 0.0
    seq = np.array([stride, stride - 3, 40001], np.int32)
    w = workloads.Workload("all_equal", "raw", k, scores, seq)
    with settings(pkg, split=split):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


# ------------------------------------------------------------ edge cases

@pytest.mark.parametrize("k", [1, 2, 7, 100, 1000, 1024, 1025, 2047, 2048])
def test_any_k(pkg, k):
    w = _mixed(300 + k, "decode", batch=4, stride=9000, k=k, form="raw")
    assert_parity(w, run_gpu(pkg, w))


@pytest.mark.parametrize("stride", [1, 2, 3, 5, 1023, 1024, 1025, 4097, 8191])
def test_odd_row_strides_and_short_rows(pkg, stride):
    """Row starts at every 4-byte alignment; L around k; L = 0; L > stride."""
    g = workloads.rng(400 + stride)
    k = 1024
    batch = 12
    scores = workloads.random_rows(g, batch, stride, "normal", dup=True)
    seq = np.array([0, 1, stride, stride + 9, -5, min(k, stride), min(k + 1, stride),
                    stride // 2, max(stride - 1, 0), 2 * stride, 3, stride], np.int32)
    for form in ("raw", "paged"):
        pt = workloads.permuted_page_table(g, batch, workloads.pages_for(stride, 64))
        w = workloads.Workload(f"stride{stride}_{form}", form, k, scores, seq, pt, 64)
        assert_parity(w, run_gpu(pkg, w))


@pytest.mark.parametrize("page_size", [1, 3, 16, 48, 64, 100, 4096])
def test_page_sizes(pkg, page_size):
    g = workloads.rng(500 + page_size)
    batch, stride, k = 4, 12000, 1024
    scores = workloads.random_rows(g, batch, stride, "heavy_tail")
    seq = np.array([stride, 5000, 800, 11999], np.int32)
    pt = workloads.permuted_page_table(g, batch, workloads.pages_for(stride, page_size))
    w = workloads.Workload(f"ps{page_size}", "paged", k, scores, seq, pt, page_size)
    assert_parity(w, run_gpu(pkg, w))


def test_identity_page_table_equals_raw(pkg):
    w = workloads.unit_test_shape(48, 32768)
    paged = run_gpu(pkg, w)
    raw = run_gpu(pkg, w.as_raw())
    assert same_sets(paged, raw).all()


@pytest.mark.parametrize("split", [1, 4, 16])
def test_ragged_odd_offsets_and_empty_rows(pkg, split):
    g = workloads.rng(600 + split)
    lens = np.array([0, 1, 2047, 2048, 2049, 70001, 3, 150000, 0, 65536], np.int64)
    gaps = g.integers(0, 7, size=lens.shape[0])
    starts = (np.concatenate([[0], np.cumsum(lens + gaps)[:-1]]) + 1).astype(np.int32)
    total = int(starts[-1] + lens[-1] + 5)
    scores = workloads.row_values(g, "banded", total, dup=True)
    w = workloads.Workload("ragged_edges", "ragged", 2048, scores, lens.astype(np.int32),
                           None, 64, starts)
    with settings(pkg, split=split):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


def test_nan_keys_follow_the_key_order(pkg):
    """NaN bit patterns are ranked by their key like any other (+NaN above +inf)."""
    g = workloads.rng(700)
    scores = workloads.random_rows(g, 2, 5000, "normal")
    scores[0, ::97] = np.float32(np.nan)
    scores[1, ::89] = -np.float32(np.nan)
    seq = np.array([5000, 5000], np.int32)
    w = workloads.Workload("nan", "raw", 1024, scores, seq)
    got = run_gpu(pkg, w)
    assert same_sets(got, oracle.run(w)).all()


def test_empty_batch(pkg):
    dev = torch.device("cuda:0")
    out = pkg.topk_transform_raw(torch.zeros((0, 16), device=dev),
                                 torch.zeros(0, dtype=torch.int32, device=dev), 4)
    assert out.shape == (0, 4)


def test_invalid_k_raises(pkg):
    dev = torch.device("cuda:0")
    s = torch.zeros((1, 16), device=dev)
    L = torch.full((1,), 16, dtype=torch.int32, device=dev)
    for k in (0, pkg.TOPK_MAX_K + 1):
        with pytest.raises(pkg.TopkError, match="unsupported k"):
            pkg.topk_transform_raw(s, L, k)


def test_side_stream_and_repeatability(pkg):
    w = workloads.config3(64, "paged")
    s = torch.cuda.Stream()
    a = run_gpu(pkg, w, stream=s)
    b = run_gpu(pkg, w)
    assert (np.sort(a, 1) == np.sort(b, 1)).all()
    assert_parity(w, a, check_rows=4)


@pytest.mark.parametrize("split", [1, 2])
def test_candidate_counts_off_block_multiples(pkg, split):
    """Rows that keep every element (length within the candidate buffer) with
    lengths just past multiples of the block size: the candidate passes must stay
    warp-uniform however many candidates there are."""
    lens = [1025, 1537, 2049, 2100, 2561, 3000, 3585, 4095, 4096]
    stride = 4200
    g = workloads.rng(900 + split)
    scores = workloads.random_rows(g, len(lens), stride, "normal", dup=True)
    seq = np.array(lens, np.int32)
    w = workloads.Workload("off_block_multiples", "raw", 1024, scores, seq)
    with settings(pkg, split=split):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


# ------------------------------------------------------------ window form (prefill-shaped rows)

def window_rows(w, rows):
    """The sub-batch of a window workload made of the given rows."""
    import dataclasses
    return dataclasses.replace(w, name=f"{w.name}_rows", scores=w.scores[rows],
                               seq_lens=w.seq_lens[rows], row_starts=w.row_starts[rows])


@pytest.mark.parametrize("window", [None, 3000, 1000])
def test_window_prefill(pkg, window):
    w = workloads.prefill_windows(512, 8192, window=window)
    assert_parity(w, run_gpu(pkg, w))


def test_window_prefill_bench_size(pkg):
    """4096 causal rows of a 32768-key context, the launch bench.py times; 256
    sampled rows against the oracle, every row through the invariant check."""
    w = workloads.prefill_windows(4096, 32768)
    got = run_gpu(pkg, w)
    rows = np.random.Generator(np.random.PCG64(3)).choice(w.batch, 256, replace=False)
    rows = np.sort(np.concatenate([rows, [0, w.batch - 1]]))
    sub = window_rows(w, rows)
    assert same_sets(got[rows], oracle.run(sub)).all()
    assert not check_workload(w, got, max_rows=None if w.batch <= 512 else 512)


def random_windows(seed, batch, stride, dist, k):
    g = np.random.Generator(np.random.PCG64(seed))
    scores = workloads.random_rows(g, batch, stride, dist, dup=True)
    starts = g.integers(-5, stride + 5, size=batch)
    ends = g.integers(-5, stride + 6, size=batch)
    # a share of long windows, so the sampled filter runs, and a few exact edges
    long_rows = g.random(batch) < 0.5
    starts[long_rows] = g.integers(-3, 9, size=int(long_rows.sum()))
    ends[long_rows] = g.integers(stride - 9, stride + 4, size=int(long_rows.sum()))
    starts[:4] = [0, stride, 3, stride - k]
    ends[:4] = [stride, stride, 2, stride]
    return workloads.Workload(f"window_random_{dist}_{stride}", "window", k, scores,
                              ends.astype(np.int32), None, 64, starts.astype(np.int32))


@pytest.mark.parametrize("split", [1, 4, 16])
@pytest.mark.parametrize("fast", [1, 0])
@pytest.mark.parametrize("dist", ["normal", "banded", "narrow"])
def test_window_random(pkg, split, fast, dist):
    w = random_windows(101 + split + 7 * fast, 48, 9001, dist, 1024)
    with settings(pkg, split=split, fast=fast):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


@pytest.mark.parametrize("tie_cap", [0, 64, 1500])
def test_window_small_tie_buffer(pkg, tie_cap):
    w = random_windows(211 + tie_cap, 24, 6007, "banded", 512)
    with settings(pkg, tie_cap=tie_cap):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


@pytest.mark.parametrize("k", [1, 5, 2048])
def test_window_any_k(pkg, k):
    w = random_windows(307 + k, 16, 5003, "heavy_tail", k)
    assert_parity(w, run_gpu(pkg, w))


def test_window_from_zero_is_raw(pkg):
    w = workloads.config3(8, "raw", c4_len=9000)
    ww = workloads.Workload("window_zero", "window", w.k, w.scores, w.seq_lens, None, 64,
                            np.zeros(w.batch, np.int32))
    assert same_sets(run_gpu(pkg, ww), run_gpu(pkg, w)).all()


# ------------------------------------------------------------ grouped calls (several problems)

def problem_of(w, dev):
    """The device-side problem dict of one workload (for topk_transform_grouped)."""
    q = {"form": w.form, "k": w.k,
         "scores": torch.from_numpy(np.ascontiguousarray(w.scores)).to(dev),
         "seq_lens": torch.from_numpy(np.ascontiguousarray(w.seq_lens)).to(dev),
         "out": torch.full((w.batch, w.k), -7, dtype=torch.int32, device=dev)}
    if w.form == "paged":
        q["page_table"] = torch.from_numpy(np.ascontiguousarray(w.page_table)).to(dev)
        q["page_size"] = w.page_size
    elif w.form == "ragged":
        q["row_starts"] = torch.from_numpy(np.ascontiguousarray(w.row_starts)).to(dev)
        q["max_row_len_hint"] = int(np.max(w.seq_lens, initial=0))
    elif w.form == "window":
        q["starts"] = torch.from_numpy(np.ascontiguousarray(w.row_starts)).to(dev)
        q["max_row_len_hint"] = w.max_row_len
    return q


def run_grouped(pkg, ws):
    dev = torch.device("cuda:0")
    outs = pkg.topk_transform_grouped([problem_of(w, dev) for w in ws])
    torch.cuda.synchronize()
    return [o.cpu().numpy() for o in outs]


def mixed_group():
    g = np.random.Generator(np.random.PCG64(5))
    raw = workloads.Workload("group_raw", "raw", 1024, workloads.random_rows(g, 8, 9001, "banded", True),
                             g.integers(0, 9100, size=8).astype(np.int32))
    small_k = workloads.config2(8192, batch=6)
    small_k.k = 7
    lens = g.integers(40000, 70000, size=3)
    starts = np.concatenate([[5], 5 + np.cumsum(lens)[:-1]]).astype(np.int32)
    packed = np.concatenate([workloads.row_values(g, "narrow", int(n), dup=True) for n in lens])
    packed = np.concatenate([np.zeros(5, np.float32), packed]).astype(np.float32)
    ragged = workloads.Workload("group_ragged", "ragged", 2048, packed, lens.astype(np.int32),
                                None, 64, starts)
    empty = workloads.Workload("group_empty", "raw", 16, np.zeros((0, 8), np.float32),
                               np.zeros(0, np.int32))
    return [workloads.config3(64), raw, workloads.prefill_windows(128, 8192, window=3000), ragged,
            empty, small_k, workloads.config5(1)]


def test_grouped_mixed_forms(pkg):
    ws = mixed_group()
    for w, got in zip(ws, run_grouped(pkg, ws)):
        if w.batch:
            assert_parity(w, got)


@pytest.mark.parametrize("split,tie_cap,fast", [(4, None, None), (None, 64, None), (None, None, 0)])
def test_grouped_settings(pkg, split, tie_cap, fast):
    ws = mixed_group()[:4]
    with settings(pkg, split=split, tie_cap=tie_cap, fast=fast):
        outs = run_grouped(pkg, ws)
    for w, got in zip(ws, outs):
        assert_parity(w, got)


def test_grouped_most_problems(pkg):
    g = np.random.Generator(np.random.PCG64(9))
    ws = []
    for i in range(pkg.TOPK_MAX_GROUP):
        B, stride = int(g.integers(1, 5)), int(g.integers(1000, 12000))
        ws.append(workloads.Workload(f"group_{i}", "raw", int(g.integers(1, 2049)),
                                     workloads.random_rows(g, B, stride, "normal"),
                                     g.integers(0, stride + 10, size=B).astype(np.int32)))
    for w, got in zip(ws, run_grouped(pkg, ws)):
        assert_parity(w, got)
    with pytest.raises(Exception):
        run_grouped(pkg, ws + ws[:1])


def test_grouped_equals_single_calls(pkg):
    w = workloads.config3(128)
    (got,) = run_grouped(pkg, [w])
    assert same_sets(got, run_gpu(pkg, w)).all()


# ------------------------------------------------------------ many rows (the 256-thread build)
# Launches of more rows than two 512-thread CTAs per SM hold (304 on 152 SMs) with
# k <= 1024 run the kernels built with 256-thread CTAs.

def many_rows(form, batch, stride, k, seed, dist="normal"):
    g = np.random.Generator(np.random.PCG64(seed))
    scores = workloads.random_rows(g, batch, stride, dist, dup=True)
    seq = g.integers(0, stride + 20, size=batch).astype(np.int32)
    seq[: batch // 2] = stride  # half the rows full length (sampled filter)
    if form == "raw":
        return workloads.Workload(f"many_raw_{batch}_{stride}", "raw", k, scores, seq)
    if form == "paged":
        pt = workloads.permuted_page_table(g, batch, workloads.pages_for(stride, 64))
        return workloads.Workload(f"many_paged_{batch}_{stride}", "paged", k, scores, seq, pt, 64)
    lens = np.minimum(seq, stride).astype(np.int64)
    starts = np.concatenate([[1], 1 + np.cumsum(lens + 3)[:-1]]).astype(np.int32)
    packed = np.zeros(int(starts[-1] + lens[-1] + 5), np.float32)
    for b in range(batch):
        packed[starts[b]:starts[b] + lens[b]] = scores[b, :lens[b]]
    return workloads.Workload(f"many_ragged_{batch}_{stride}", "ragged", k, packed,
                              lens.astype(np.int32), None, 64, starts)


@pytest.mark.parametrize("form", ["raw", "paged", "ragged"])
@pytest.mark.parametrize("fast", [1, 0])
def test_many_rows(pkg, form, fast):
    w = many_rows(form, 400, 8192, 1024, 41 + fast, "banded" if fast else "normal")
    with settings(pkg, fast=fast):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


def test_many_long_paged_rows(pkg):
    """Rows of more pages than the 256-thread build stages (1024): the page table is
    read from global memory."""
    w = many_rows("paged", 320, 70000, 1024, 43)
    assert_parity(w, run_gpu(pkg, w))


@pytest.mark.parametrize("tie_cap", [0, 64, 4096])
def test_many_rows_tie_capacity(pkg, tie_cap):
    w = many_rows("raw", 320, 6000, 700, 47 + tie_cap, "narrow")
    with settings(pkg, tie_cap=tie_cap):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


@pytest.mark.parametrize("k", [1, 1024, 1025])
def test_many_rows_k_switches_build(pkg, k):
    w = many_rows("raw", 330, 5000, k, 53)
    assert_parity(w, run_gpu(pkg, w))


def test_grouped_many_rows(pkg):
    ws = [many_rows("raw", 40, 4096 + 512 * i, 1024, 60 + i) for i in range(12)]
    for w, got in zip(ws, run_grouped(pkg, ws)):
        assert_parity(w, got)


# ------------------------------------------------------------ the 256-thread build on every path

@pytest.mark.parametrize("fast", [True, False])
@pytest.mark.parametrize("split", [1, 4, 16])
@pytest.mark.parametrize("dist", ["normal", "decode", "banded", "narrow", "subnormal", "heavy_tail"])
def test_every_row_split_cta256(pkg, split, dist, fast):
    w = _mixed(100 + split, dist)
    with settings(pkg, split=split, fast=fast, cta=256):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


@pytest.mark.parametrize("tie_cap", [0, 16, 300, 3072, 4096])
@pytest.mark.parametrize("split", [1, 4])
@pytest.mark.parametrize("dist", ["decode", "banded", "narrow", "subnormal"])
def test_tie_buffer_capacity_cta256(pkg, tie_cap, split, dist):
    w = _mixed(200 + tie_cap, dist, k=2048)
    with settings(pkg, split=split, tie_cap=tie_cap, cta=256):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


def pages_workloads():
    return [workloads.config1(), workloads.config2(8192), workloads.config2(32768),
            workloads.config3(64), workloads.config3(256, "raw"), workloads.config4("banded"),
            workloads.config5(1), workloads.prefill_windows(256, 8192, window=2000)]


@pytest.mark.parametrize("cta", [256, 512])
def test_pages_workloads_on_each_build(pkg, cta):
    for w in pages_workloads():
        with settings(pkg, cta=cta):
            got = run_gpu(pkg, w)
        assert_parity(w, got, check_rows=8)


@pytest.mark.parametrize("split", [1, 16])
def test_all_equal_rows_cta256(pkg, split):
    batch, stride, k = 3, 50000, 2048
    scores = np.full((batch, stride), 1.5, np.float32)
    scores[1, ::7] = -0.0
    scores[2] = 0.0
    seq = np.array([stride, stride - 3, 40001], np.int32)
    w = workloads.Workload("all_equal_cta256", "raw", k, scores, seq)
    with settings(pkg, split=split, cta=256):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


# ------------------------------------------------------------ values and sorted output

def run_options(pkg, ws, sorted_=False, static_workspace=False):
    """Grouped call with the values output (and the sorted option) on every problem."""
    dev = torch.device("cuda:0")
    probs = []
    for w in ws:
        q = problem_of(w, dev)
        q["values"] = torch.full((w.batch, w.k), 7.0, dtype=torch.float32, device=dev)  # poison
        q["sorted"] = sorted_
        probs.append(q)
    outs = pkg.topk_transform_grouped(probs, static_workspace=static_workspace)
    torch.cuda.synchronize()
    return [(o.cpu().numpy(), q["values"].cpu().numpy()) for o, q in zip(outs, probs)]


def assert_options(w, got, vals, sorted_):
    exp, exp_vals = oracle.run_values(w)
    if sorted_:  # rank order and values, slot by slot
        bad = np.flatnonzero(~(got == exp).all(axis=1))
        assert bad.size == 0, f"{w.name}: row {bad[0]} order {got[bad[0]][:8]} vs {exp[bad[0]][:8]}"
        assert (vals.view(np.uint32) == exp_vals.view(np.uint32)).all(), f"{w.name}: values differ"
    else:  # the set, and each slot's value belongs to its position
        assert_parity(w, got)
        order_got, order_exp = np.argsort(got, axis=1), np.argsort(exp, axis=1)
        v_got = np.take_along_axis(vals, order_got, 1).view(np.uint32)
        v_exp = np.take_along_axis(exp_vals, order_exp, 1).view(np.uint32)
        assert (v_got == v_exp).all(), f"{w.name}: values do not follow their positions"


def option_workloads():
    g = np.random.Generator(np.random.PCG64(71))
    ties = workloads.Workload("opt_ties", "raw", 300, np.round(
        workloads.random_rows(g, 5, 3000, "normal"), 1).astype(np.float32),
        np.array([3000, 2999, 200, 0, 2500], np.int32))
    return [workloads.config1(), workloads.config2(8192, batch=12), workloads.config3(8, "raw"),
            workloads.config4("narrow", batch=3), workloads.prefill_windows(64, 4096, window=1500),
            ties, workloads.config5(1)]


@pytest.mark.parametrize("sorted_", [False, True])
def test_values_and_sorted_output(pkg, sorted_):
    ws = option_workloads()
    for w, (got, vals) in zip(ws, run_options(pkg, ws, sorted_)):
        assert_options(w, got, vals, sorted_)


@pytest.mark.parametrize("staged", [2, 3])
@pytest.mark.parametrize("sorted_", [False, True])
def test_values_and_sorted_output_staged(pkg, sorted_, staged):
    """The options (values, rank order) through grouped launches on the staged tier."""
    ws = option_workloads()
    with settings(pkg, staged=staged):
        outs = run_options(pkg, ws, sorted_)
    for w, (got, vals) in zip(ws, outs):
        assert_options(w, got, vals, sorted_)


@pytest.mark.parametrize("cta", [256, 512])
@pytest.mark.parametrize("fast", [1, 0])
@pytest.mark.parametrize("split", [1, 4])
def test_sorted_output_every_path(pkg, cta, fast, split):
    ws = [_mixed(300 + split, "banded", batch=4), _mixed(301, "narrow", batch=3, k=2048),
          many_rows("paged", 40, 5000, 1000, 73)]
    with settings(pkg, cta=cta, fast=fast, split=split):
        outs = run_options(pkg, ws, True)
    for w, (got, vals) in zip(ws, outs):
        assert_options(w, got, vals, True)


@pytest.mark.parametrize("k", [1, 2, 1023, 2048])
def test_sorted_any_k(pkg, k):
    w = many_rows("raw", 6, 9000, k, 80 + k, "heavy_tail")
    ((got, vals),) = run_options(pkg, [w], True)
    assert_options(w, got, vals, True)


def test_sorted_output_static_workspace(pkg):
    """The call that stages in the library's own scratch array: same results; twice
    in a row on one stream (the array is reused)."""
    ws = option_workloads()
    for _ in range(2):
        for w, (got, vals) in zip(ws, run_options(pkg, ws, True, static_workspace=True)):
            assert_options(w, got, vals, True)


def test_static_workspace_too_small(pkg):
    dev = torch.device("cuda:0")
    B, k = (16 << 20) // (8 * 2048) + 1, 2048
    w = workloads.Workload("too_big", "raw", k, np.zeros((B, 8), np.float32),
                           np.full(B, 8, np.int32))
    q = problem_of(w, dev)
    q["sorted"] = True
    with pytest.raises(pkg.TopkError):
        pkg.topk_transform_grouped([q], static_workspace=True)


# ------------------------------------------------------------ graphs and streams

def test_calls_captured_in_a_cuda_graph(pkg):
    """Calls of every form captured in one CUDA graph (launches with programmatic
    dependencies between them) and replayed give the oracle's results."""
    dev = torch.device("cuda:0")
    ws = [workloads.config3(64), workloads.config3(8, "raw"), workloads.config4("subnormal", batch=2),
          workloads.prefill_windows(300, 6000, window=2500)]
    probs = [problem_of(w, dev) for w in ws]
    sorted_q = problem_of(workloads.config2(8192, batch=5), dev)
    sorted_q["sorted"] = True
    sorted_q["values"] = torch.empty((5, 1024), dtype=torch.float32, device=dev)
    sort_ws = torch.empty(5 * 1024 * 8, dtype=torch.uint8, device=dev)  # allocated before capture
    stream = torch.cuda.Stream(dev)

    def calls():
        for w, q in zip(ws, probs):
            if w.form == "paged":
                pkg.topk_transform_paged(q["scores"], q["seq_lens"], q["page_table"], w.page_size,
                                         w.k, out=q["out"], stream=stream)
            elif w.form == "raw":
                pkg.topk_transform_raw(q["scores"], q["seq_lens"], w.k, out=q["out"], stream=stream)
            elif w.form == "ragged":
                pkg.topk_transform_ragged(q["scores"], q["row_starts"], q["seq_lens"], w.k,
                                          max_row_len_hint=q["max_row_len_hint"], out=q["out"],
                                          stream=stream)
            else:
                pkg.topk_transform_window(q["scores"], q["starts"], q["seq_lens"], w.k,
                                          max_row_len_hint=q["max_row_len_hint"], out=q["out"],
                                          stream=stream)
        pkg.topk_transform_grouped([sorted_q], stream=stream, workspace=sort_ws)

    with torch.cuda.stream(stream):
        calls()  # first calls set the device up outside the capture
        stream.synchronize()
        for q in probs + [sorted_q]:
            q["out"].fill_(-7)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            calls()
        for _ in range(3):
            graph.replay()
        stream.synchronize()
    for w, q in zip(ws, probs):
        assert_parity(w, q["out"].cpu().numpy())
    w2 = workloads.config2(8192, batch=5)
    assert_options(w2, sorted_q["out"].cpu().numpy(), sorted_q["values"].cpu().numpy(), True)


def test_concurrent_streams(pkg):
    """Two streams running different problems at the same time."""
    dev = torch.device("cuda:0")
    wa, wb = workloads.config3(128), many_rows("raw", 320, 7000, 900, 91)
    qa, qb = problem_of(wa, dev), problem_of(wb, dev)
    sa, sb = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    torch.cuda.synchronize()
    for _ in range(3):
        pkg.topk_transform_paged(qa["scores"], qa["seq_lens"], qa["page_table"], wa.page_size, wa.k,
                                 out=qa["out"], stream=sa)
        pkg.topk_transform_raw(qb["scores"], qb["seq_lens"], wb.k, out=qb["out"], stream=sb)
    torch.cuda.synchronize()
    assert_parity(wa, qa["out"].cpu().numpy())
    assert_parity(wb, qb["out"].cpu().numpy())


# ------------------------------------------------------------ the filter-time L1 read-back
# Single-CTA launches of more rows than SMs (152) with the 512-thread build read the
# candidates' values back from L1 inside the filter.

def special_rows(g, batch, stride):
    """Rows mixing NaN of both signs, infinities, signed zeros, subnormals, exact
    duplicates and ordinary values."""
    x = workloads.random_rows(g, batch, stride, "normal", dup=True)
    pick = g.random(x.shape)
    x[pick < 0.01] = np.float32(np.nan)
    x[(pick >= 0.01) & (pick < 0.02)] = -np.float32(np.nan)
    x[(pick >= 0.02) & (pick < 0.03)] = np.float32(np.inf)
    x[(pick >= 0.03) & (pick < 0.04)] = -np.float32(np.inf)
    x[(pick >= 0.04) & (pick < 0.06)] = np.float32(0.0)
    x[(pick >= 0.06) & (pick < 0.08)] = -np.float32(0.0)
    x[(pick >= 0.08) & (pick < 0.10)] = np.float32(1e-40)
    return x


@pytest.mark.parametrize("stride", [3000, 20000])
@pytest.mark.parametrize("form", ["raw", "paged", "ragged"])
def test_keys_in_filter_special_values(pkg, stride, form):
    """Short rows (every element a candidate, no sample) and sampled rows, with special
    values, at a batch that takes the L1 read-back (and paged with a page size that
    is not a power of two)."""
    g = np.random.Generator(np.random.PCG64(stride + len(form)))
    batch, k = 200, 1024
    scores = special_rows(g, batch, stride)
    seq = g.integers(0, stride + 5, size=batch).astype(np.int32)
    seq[::3] = stride
    if form == "raw":
        w = workloads.Workload(f"keys_raw_{stride}", "raw", k, scores, seq)
    elif form == "paged":
        pt = workloads.permuted_page_table(g, batch, workloads.pages_for(stride, 48))
        w = workloads.Workload(f"keys_paged_{stride}", "paged", k, scores, seq, pt, 48)
    else:
        lens = np.minimum(seq, stride).astype(np.int64)
        starts = np.concatenate([[7], 7 + np.cumsum(lens + 1)[:-1]]).astype(np.int32)
        packed = np.zeros(int(starts[-1] + lens[-1] + 3), np.float32)
        for b in range(batch):
            packed[starts[b]:starts[b] + lens[b]] = scores[b, :lens[b]]
        w = workloads.Workload(f"keys_ragged_{stride}", "ragged", k, packed,
                               lens.astype(np.int32), None, 64, starts)
    got = run_gpu(pkg, w)
    exp = oracle.run(w)
    assert same_sets(got, exp).all(), f"{w.name}: rows differ from the oracle"


@pytest.mark.parametrize("tie_cap", [0, 300, 4096])
def test_keys_in_filter_tie_capacity(pkg, tie_cap):
    w = many_rows("paged", 200, 12000, 1024, 97 + tie_cap, "banded")
    with settings(pkg, tie_cap=tie_cap):
        got = run_gpu(pkg, w)
    assert_parity(w, got)


# ------------------------------------------------------------ threshold-bin sizes
# The candidates of the threshold bin are ordered by a direct rank count up to the
# CTA size and by radix rounds beyond it.

def threshold_bin_rows(batch, stride, k, dup, seed):
    """Rows whose k-th score is repeated `dup` times (the repeats straddle rank k),
    so the threshold bin holds at least `dup` equal keys; some rows centre the
    scores near zero, where the key jumps across the sign."""
    g = workloads.rng(seed)
    scores = workloads.random_rows(g, batch, stride, "normal")
    for b in range(batch):
        row = scores[b]
        if b % 2 == 1:
            row -= np.float32(1.86)  # the k-th score near zero
        order = np.argsort(-row, kind="stable")
        v = row[order[k - 1 - dup // 2]]
        pos = g.choice(stride, size=dup, replace=False)
        row[pos] = v
    return scores


@pytest.mark.parametrize("cta", [512, 256])
@pytest.mark.parametrize("dup", [1, 2, 3, 63, 64, 65, 127, 128, 129, 200, 256, 257, 512, 513, 900])
def test_threshold_bin_sizes(pkg, dup, cta):
    batch, stride, k = 6, 32768, 1024
    scores = threshold_bin_rows(batch, stride, k, dup, 1300 + dup)
    seq = np.full(batch, stride, np.int32)
    w = workloads.Workload(f"tbin_{dup}", "raw", k, scores, seq)
    with settings(pkg, cta=cta, split=1):
        assert_parity(w, run_gpu(pkg, w))
    with settings(pkg, cta=cta, split=4):
        assert_parity(w, run_gpu(pkg, w))
