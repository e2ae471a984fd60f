"""The roofline cost model behind LCGEMM_AUTO, through a planning handle (CPU only, no CUDA call)."""
import pytest

import complexity_matmul_gb300 as lcg
from complexity_matmul_gb300 import _build


@pytest.fixture(scope="module")
def plan():
    _build.build()
    h = lcg.Handle(lcg.PLANNING_DEVICE)
    yield h
    h.close()


def test_planning_handle_rejects_runs(plan):
    assert plan.run_raw(8, 8, 8, None, 8, None, 8, None, 8, lcg.BF16, lcg.PLAIN) == lcg.ERR_ARG
    assert plan.sync_status() == lcg.ERR_ARG


def test_non_divisible_shapes_pay_for_padding(plan):
    # one level pads M, N to even and K to a multiple of 16; two levels to multiples of 4 and 32
    t_even = plan.estimate(8192, 8192, 8192, lcg.BF16, "strassen1")
    t_odd = plan.estimate(8191, 8193, 8190, lcg.BF16, "strassen1")
    assert t_odd > t_even
    # the padding costs one read and one write of A and B at HBM speed, far below the GEMM itself
    assert t_odd < t_even * 1.2
    assert plan.estimate(131, 66, 48, lcg.BF16, "strassen1") > 0
    assert plan.estimate(130, 68, 64, lcg.BF16, "strassen2") > plan.estimate(132, 68, 64, lcg.BF16, "strassen2")
    assert plan.estimate(0, 8, 8, lcg.BF16, "strassen1") == 0.0      # an empty C: nothing runs


@pytest.mark.parametrize("shape", [(131, 257, 1000), (1, 4096, 4095), (4097, 4097, 4097), (64, 64, 8)])
def test_auto_never_picks_an_unsupported_algorithm(plan, shape):
    assert plan.select(*shape, lcg.BF16) == lcg.PLAIN


def test_plain_estimate_grows_with_work(plan):
    prev = 0.0
    for n in (256, 1024, 2048, 4096, 8192, 16384):
        t = plan.estimate(n, n, n, lcg.BF16, "plain")
        assert t > prev
        prev = t
    # a compute-bound square GEMM runs within 2x of the tensor peak it is given
    t = plan.estimate(16384, 16384, 16384, lcg.BF16, "plain")
    assert 2 * 16384 ** 3 / 2.25e15 < t < 2 * 2 * 16384 ** 3 / 2.25e15


def test_skinny_gemm_is_bandwidth_bound(plan):
    M, N, K = 1, 14336, 4096
    t = plan.estimate(M, N, K, lcg.BF16, "plain")
    compulsory = 2.0 * (M * K + K * N + M * N) / 8e12
    assert compulsory < t < 3 * compulsory


def test_wave_quantisation():
    """76 CTA pairs of 256x256 tiles: 80 tiles cost a second wave (or half of one when the
    partial last wave is split into K halves)."""
    h = lcg.Handle(lcg.PLANNING_DEVICE)
    K = 16384
    full = h.estimate(1024, 256 * 19, K, lcg.BF16, "plain")     # 76 tiles: one full wave
    over = h.estimate(1024, 256 * 20, K, lcg.BF16, "plain")     # 80 tiles
    assert 1.3 * full < over < 1.7 * full
    h.set_option(lcg.OPT_SPLIT, 0)
    over_nosplit = h.estimate(1024, 256 * 20, K, lcg.BF16, "plain")
    assert over_nosplit > 1.7 * full
    h.close()


def test_tail_split_from_48_slabs(plan):
    """The partial last wave runs as K halves from 48 K slabs (K = 3072): 80 tiles then cost about
    one and a half waves of 76; with 32 slabs (K = 2048) the exchange does not pay, and the model
    prices 80 tiles as with the split switched off."""
    split, nosplit = lcg.Handle(lcg.PLANNING_DEVICE), lcg.Handle(lcg.PLANNING_DEVICE)
    for h in (split, nosplit):
        h.set_option(lcg.OPT_PLAIN_KERNEL, 2)        # 256 x 256 pair tiles
    nosplit.set_option(lcg.OPT_SPLIT, 0)

    def ratio(h, K):
        return h.estimate(1024, 256 * 20, K, lcg.BF16, "plain") / h.estimate(1024, 256 * 19, K, lcg.BF16, "plain")
    for K in (3072, 4096, 6144):
        assert ratio(split, K) < 1.7 < ratio(nosplit, K)
    assert ratio(split, 2048) == pytest.approx(ratio(nosplit, 2048))
    split.close()
    nosplit.close()


def test_pair_tile_width():
    """256 x 512 pair tiles when their wave-quantised time, with ~10 slabs of epilogue per wide tile
    and less the wide tiles' measured 8 % per unit of work, beats 256 x 256 tiles: the long main
    loops of 16384^3 (27 waves against 54), 12288^3 and 8192^3 take them; the shapes where they
    measured slower do not: K = 4096 (1024x14336, 4096x16384: 3-8 % slower), a split wide tail
    against one narrow wave (1024x4096x14336), 4096^3 and 2048^3.  The model prices whichever the
    dispatcher takes."""
    wide, narrow, auto = (lcg.Handle(lcg.PLANNING_DEVICE) for _ in range(3))
    wide.set_option(lcg.OPT_PLAIN_KERNEL, 5)
    narrow.set_option(lcg.OPT_PLAIN_KERNEL, 2)
    cases = [((16384, 16384, 16384), wide), ((12288, 12288, 12288), wide), ((8192, 8192, 8192), wide),
             ((1024, 14336, 4096), narrow), ((4096, 16384, 4096), narrow), ((1024, 4096, 14336), narrow),
             ((4096, 4096, 4096), narrow), ((2048, 2048, 2048), narrow)]
    for (m, n, k), want in cases:
        t = auto.estimate(m, n, k, lcg.BF16, "plain")
        assert t == pytest.approx(want.estimate(m, n, k, lcg.BF16, "plain")), (m, n, k)
        other = narrow if want is wide else wide
        assert t < other.estimate(m, n, k, lcg.BF16, "plain"), (m, n, k)
    for h in (wide, narrow, auto):
        h.close()


def test_strassen_saves_multiplies_only_when_large(plan):
    # small shapes: the pre-pass and launches dominate, plain wins
    for n in (256, 1024, 2048):
        assert plan.select(n, n, n, lcg.BF16) == lcg.PLAIN
        assert plan.estimate(n, n, n, lcg.BF16, "strassen1") > plan.estimate(n, n, n, lcg.BF16, "plain")
    # the one-level model charges 7/8 of the multiplications plus 4.5(MK+KN) bytes of pre-pass
    n = 65536
    t1 = plan.estimate(n, n, n, lcg.BF16, "strassen1")
    t0 = plan.estimate(n, n, n, lcg.BF16, "plain")
    assert t1 < 1.2 * t0


def test_peak_and_bandwidth_options_move_the_choice(plan):
    h = lcg.Handle(lcg.PLANNING_DEVICE)
    n = 32768
    base = h.estimate(n, n, n, lcg.BF16, "plain")
    h.set_option(lcg.OPT_PEAK_GFLOPS, 4_500_000)     # twice the tensor peak: compute time halves
    assert h.estimate(n, n, n, lcg.BF16, "plain") < 0.6 * base
    h.set_option(lcg.OPT_HBM_GBPS, 100)              # starve the bandwidth: the pre-pass dominates
    assert h.select(n, n, n, lcg.BF16) == lcg.PLAIN
    with pytest.raises(lcg.LcgemmError):
        h.set_option(lcg.OPT_PEAK_GFLOPS, 0)
    h.close()


def test_few_tile_long_k_shapes_use_split_k(plan):
    """A 128 x 512 output with K = 16384 has two 128 x 256 tiles: the model spreads them over the
    machine as split-K work items (measured ~25 us on GB300), not two CTAs walking 256 K slabs."""
    M, N, K = 128, 512, 16384
    t = plan.estimate(M, N, K, lcg.BF16, "plain")
    one_cta_per_tile = 2.0 * M * N * K / (2.25e15 / 152)          # two tiles, one SM each
    assert t < 0.5 * one_cta_per_tile
    assert t < plan.estimate(M, N, K, lcg.BF16, "strassen2")
    assert plan.select(M, N, K, lcg.BF16) == lcg.PLAIN


def test_split_k_threshold_at_48_slabs(plan):
    """Split-K starts at 48 K slabs: a 32-slab tile runs unsplit (two 16-slab chunks measured 3 us
    slower than one CTA on GB300), while 48 slabs split into three chunks, so at M = 16 (chunks
    summed by the last to arrive, no extra launch) the longer K is estimated cheaper."""
    t32 = plan.estimate(16, 256, 2048, lcg.BF16, "plain")
    t48 = plan.estimate(16, 256, 3072, lcg.BF16, "plain")
    assert t48 < t32      # were 32 slabs split too, both would run 16-slab chunks


def test_pair_tiles_only_when_they_fill_the_pairs(plan):
    """CTA pairs need their 256 x 256 tiles to fill a quarter of the pairs; below that the estimate
    is the single-CTA split-K one, which for few tiles is lower than the pair estimate."""
    h = lcg.Handle(lcg.PLANNING_DEVICE)
    shape = (256, 4096, 14336)                     # 16 pair tiles on 76 pairs
    t_default = h.estimate(*shape, lcg.BF16, "plain")
    h.set_option(lcg.OPT_PLAIN_KERNEL, 2)
    t_pair = h.estimate(*shape, lcg.BF16, "plain")
    h.close()
    assert t_default < t_pair


def test_degenerate_shapes(plan):
    """An empty C launches nothing (estimate 0); K = 0 still writes C (a launch); negative sizes,
    unknown dtypes and unknown algorithms are argument errors."""
    import ctypes
    def est(M, N, K, dtype=lcg.BF16, algo=lcg.PLAIN):
        s = ctypes.c_double(-1.0)
        return plan._lib.lcgemm_estimate(plan._h, M, N, K, dtype, algo, ctypes.byref(s)), s.value
    assert est(0, 128, 128) == (lcg.OK, 0.0)
    assert est(128, 0, 128, algo=lcg.STRASSEN2) == (lcg.OK, 0.0)
    rc, t = est(128, 128, 0)
    assert rc == lcg.OK and t > 0.0
    assert est(128, 128, 0, algo=lcg.STRASSEN1) == (rc, t)        # K = 0 fills C the same way
    assert est(-1, 128, 128)[0] == lcg.ERR_ARG
    assert est(128, 128, 128, dtype=7)[0] == lcg.ERR_ARG
    assert est(128, 128, 128, algo=9)[0] == lcg.ERR_ARG


def _h20_like():
    """A bandwidth-rich, compute-poor part like the write-up's H20 (about 148 TFLOP/s dense FP16,
    4 TB/s HBM, 78 SMs): FalconGEMM write-up, section "从 LCMA 到 FalconGEMM" (H20 suits trading
    extra data handling for fewer multiplications) and "从缓存重排到 Cost Model" (LCMA only pays
    where the GEMM is compute-bound)."""
    h = lcg.Handle(lcg.PLANNING_DEVICE)
    h.set_option(lcg.OPT_PEAK_GFLOPS, 148_000)
    h.set_option(lcg.OPT_HBM_GBPS, 4_000)
    h.set_option(lcg.OPT_MAX_CTAS, 78)
    return h


def test_h20_like_machine_picks_strassen_only_for_large_cubes():
    """On a machine with ~15x less tensor throughput per byte of bandwidth the model must pick
    Strassen for large compute-bound cubes and keep plain for the shapes where the
    pre-pass or the per-product pipeline refills outweigh the 1/8 of multiplications saved.
    A Strassen efficiency that cannot reach 7/8 of plain's never picks it (first assertion);
    a model without the refill cost picks it at 8192^3 too (second)."""
    h = _h20_like()
    for n in (16384, 20480):
        assert h.select(n, n, n, lcg.BF16) in (lcg.STRASSEN1, lcg.STRASSEN2), n
    # a second level pays once the cube is large enough to amortise its larger pre-pass
    assert h.select(24576, 24576, 24576, lcg.BF16) == lcg.STRASSEN2
    for n in (2048, 4096, 8192):
        assert h.select(n, n, n, lcg.BF16) == lcg.PLAIN, n
    # 12288^3 sits at the crossover (plain's 256 x 512 tiles within 2 % of one level)
    t = {a: h.estimate(12288, 12288, 12288, lcg.BF16, a) for a in ("plain", "strassen1")}
    assert abs(t["plain"] / t["strassen1"] - 1) < 0.05
    h.close()


def test_gb300_model_keeps_plain_on_the_measured_shapes(plan):
    """On GB300 the plain CTA-pair kernel was the fastest algorithm on every shape measured (the
    square sweep, the large rectangles, all 1000 grid shapes): the model must not pick Strassen
    there.  A model that drops the per-product refill cost picks strassen1 at 16384^3."""
    import synthetic
    for n in (2048, 4096, 8192, 16384):
        assert plan.select(n, n, n, lcg.BF16) == lcg.PLAIN, n
    for shape in synthetic.LARGE_RECT:
        assert plan.select(*shape, lcg.BF16) == lcg.PLAIN, shape
    picks = [plan.select(M, N, K, lcg.F16) for (M, N, K) in synthetic.grid_triples()]
    assert picks.count(lcg.PLAIN) == len(picks)


def test_prepass_is_priced_at_streaming_bandwidth(plan):
    """The Combine-A/B pre-pass reads A and B once and writes five summed blocks of each (the
    other two products read raw blocks in place): 4.5 bytes per element of A and B, priced at the
    model's streaming fraction (0.8) of the HBM bandwidth.  Removing the bandwidth (1e9 GB/s)
    removes exactly that time from a compute-bound one-level estimate."""
    h = lcg.Handle(lcg.PLANNING_DEVICE)
    M, N, K = 16384, 16384, 16384
    t_bw = h.estimate(M, N, K, lcg.BF16, "strassen1")
    h.set_option(lcg.OPT_HBM_GBPS, 1_000_000_000)
    t_inf = h.estimate(M, N, K, lcg.BF16, "strassen1")
    h.close()
    expect = 4.5 * (M * K + K * N) / (0.8 * 8000e9)
    assert abs((t_bw - t_inf) - expect) < 0.02 * expect
