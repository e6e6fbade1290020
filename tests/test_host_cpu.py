"""CPU-only checks: the C-ABI library loads and exports every symbol its
header declares, host-side argument checks reject bad configurations before
touching CUDA, and the benchmark's host logic (byte counts, clock parsing,
multi-rank aggregation over gloo) is right."""
import ctypes
import os
import re

import pytest

import bench
import speculative_decoding_verification_22_gb300 as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            text = open(os.path.join(inc, fn)).read()
            names.update(re.findall(r"^[\w\s\*]*?\b(spec_\w+)\s*\(", text, re.M))
    return names


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_22_gb300 import build as b
    b.build()
    return sv.load_library()


def test_library_exports_every_header_symbol(lib):
    names = header_symbols()
    assert len(names) >= 13
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing
    assert set(names) == set(sv.EXPORTS)


def test_strerror_covers_every_code(lib):
    for code in range(0, -9, -1):
        assert sv.spec_verify_strerror(code) != "unknown error"
    assert sv.spec_verify_strerror(-99) == "unknown error"


@pytest.mark.parametrize("cfg,want", [
    (dict(V=0, d=4096, B=1, K=4, dtype=0), sv.SV_ERR_SHAPE),
    (dict(V=128256, d=4095, B=1, K=4, dtype=0), sv.SV_ERR_SHAPE),   # d % 8
    (dict(V=128256, d=4096, B=0, K=4, dtype=0), sv.SV_ERR_SHAPE),
    (dict(V=128256, d=4096, B=1, K=65, dtype=0), sv.SV_ERR_SHAPE),  # K > 64
    (dict(V=128256, d=4096, B=65, K=5, dtype=0), sv.SV_ERR_SHAPE),  # 390 rows
    (dict(V=1000, d=256, B=1, K=4, dtype=7), sv.SV_ERR_ARG),
    (dict(V=1000, d=6, B=1, K=4, dtype=1), sv.SV_ERR_SHAPE),        # d % 4
])
def test_create_rejects_bad_configurations_before_cuda(lib, cfg, want):
    c = sv.sv_config_t(cfg["V"], cfg["d"], cfg["B"], cfg["K"], cfg["dtype"], None)
    h = ctypes.c_void_p(1)
    assert lib.spec_verify_create(ctypes.byref(c), ctypes.byref(h)) == want
    assert not h.value


def test_null_arguments_are_rejected(lib):
    assert lib.spec_verify_create(None, None) == sv.SV_ERR_ARG
    assert lib.spec_verify_run(None, None, None, None, None, None, 1.0, None, None) == sv.SV_ERR_ARG
    assert lib.spec_verify_status(None) == sv.SV_ERR_ARG
    lib.spec_verify_destroy(None)


def test_algorithmic_bytes_of_the_llama8b_round():
    # W_lm + q_logits + hidden + tokens + uniforms + outputs at V=128256,
    # d=4096, B=1, K=4
    assert bench.algorithmic_bytes(128256, 4096, 1, 4) == 1_052_766_268
    assert bench.contraction_bytes(128256, 4096, 1, 4) == (2 * 128256 * 4096 + 2 * 5 * 4096
                                                           + 4 * 4 * 128256)
    greedy = bench.algorithmic_bytes(128256, 4096, 8, 7, greedy=True)
    assert greedy == 2 * 128256 * 4096 + 2 * 64 * 4096 + 4 * 56 + 4 * 64 + 4 * 8


def test_input_sets_exceed_l2():
    n = bench.n_input_sets(2_100_000)
    assert n * 2_100_000 >= 2 * bench.L2_BYTES
    assert bench.n_input_sets(10 ** 10) == 4


def test_parse_clocks():
    text = ("index, clocks.sm [MHz], clocks.max.sm [MHz], power.draw [W], "
            "clocks_event_reasons.active, clocks_event_reasons.hw_slowdown, "
            "clocks_event_reasons.hw_thermal_slowdown, clocks_event_reasons.sw_thermal_slowdown, "
            "clocks_event_reasons.sw_power_cap\n"
            "0, 1965 MHz, 2070 MHz, 900.1 W, 0x0000, Not Active, Not Active, Not Active, Not Active\n"
            "0, 1800 MHz, 2070 MHz, 1300.0 W, 0x0004, Not Active, Not Active, Not Active, Active\n"
            "0, 345 MHz, 2070 MHz, 150.0 W, 0x0001, Not Active, Not Active, Not Active, Not Active\n")
    c = bench.parse_clocks(text)
    assert c["sm_max_mhz"] == 2070
    # nvidia-smi labels the queried clocks.sm column clocks.current.sm
    c2 = bench.parse_clocks(text.replace("clocks.sm [MHz]", "clocks.current.sm [MHz]", 1))
    assert c2 == c
    assert c["sm_mhz"] == pytest.approx((1965 + 1800) / 2)
    assert c["reasons"] == ["sw_power_cap"]


def _gloo_worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.aggregate(0.5 + rank, 100 + rank)))
    finally:
        dist.destroy_process_group()


def test_rank_aggregation_over_gloo():
    import multiprocessing as mp
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_gloo_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        assert results[r] == (1.5, 201)


def test_ngram_draft_rejects_bad_arguments_before_cuda(lib):
    f = lib.spec_ngram_draft
    good = 1 << 12  # aligned fake addresses: the checks never dereference
    assert f(None, 8, good, 1, 4, 2, 5, good, good, None) == sv.SV_ERR_ARG
    assert f(good, 8, good, 0, 4, 2, 5, good, good, None) == sv.SV_ERR_ARG    # B
    assert f(good, 0, good, 1, 4, 2, 5, good, good, None) == sv.SV_ERR_ARG    # ld
    assert f(good, 8, good, 1, 0, 2, 5, good, good, None) == sv.SV_ERR_ARG    # K
    assert f(good, 8, good, 1, 65, 2, 5, good, good, None) == sv.SV_ERR_ARG   # K > 64
    assert f(good, 8, good, 1, 4, 0, 5, good, good, None) == sv.SV_ERR_ARG    # n_min
    assert f(good, 8, good, 1, 4, 3, 2, good, good, None) == sv.SV_ERR_ARG    # n_max < n_min
    assert f(good, 8, good, 1, 4, 2, 17, good, good, None) == sv.SV_ERR_ARG   # n_max > 16
    assert f(good + 2, 8, good, 1, 4, 2, 5, good, good, None) == sv.SV_ERR_ALIGN


def test_sweep_points_cover_the_batch_grid():
    pts = bench.sweep_points()
    assert len(pts) == 21
    assert (1, 3) in pts and (64, 5) in pts
    assert bench.sweep_points("16x4,64X5") == [(16, 4), (64, 5)]


def test_sweep_regime_follows_the_larger_fraction():
    assert bench.regime(0.9, 0.1) == "hbm"
    assert bench.regime(0.4, 0.7) == "tensor"


SMEM_OPTIN = 232448   # opt-in shared memory per block on GB300
TMEM_COLS = 512


def _plans():
    for dtype in ("bf16", "fp8"):
        for V, d in ((128256, 4096), (128256, 8192), (1000, 960), (33, 256)):
            if dtype == "fp8" and d % 16:
                continue
            for B in range(1, 65):
                for K in range(0, 8):
                    if B * (K + 1) > sv.SV_MAX_ROWS_BF16:
                        continue
                    yield dtype, V, d, B, K, sv.spec_verify_plan(V, d, B, K, dtype)


def test_contraction_plan_fits_the_gpu_for_every_shape(lib):
    n = 0
    for dtype, V, d, B, K, p in _plans():
        n += 1
        R = B * (K + 1)
        npad_all = (R + 15) // 16 * 16
        where = (dtype, V, d, B, K, p)
        # shared memory: at least two stages, within the opt-in limit
        assert p["stages"] >= 2 and p["smem_bytes"] <= SMEM_OPTIN, where
        assert p["stage_bytes"] % 1024 == 0, where
        assert p["stages"] * p["stage_bytes"] < p["smem_bytes"], where
        # k blocks: 128-byte rows, whole chunks per stage
        assert p["kblock_elems"] * (1 if dtype == "fp8" else 2) == 128, where
        assert p["kblocks"] == -(-d // p["kblock_elems"]) and p["kblocks"] % p["chunks"] == 0
        # tensor memory: a power-of-two allocation holding every accumulator
        cols = p["tmem_cols"]
        assert 32 <= cols <= TMEM_COLS and cols & (cols - 1) == 0, where
        if p["drain_cols"]:
            # drain mode up to 64 columns: a ring of slots of its width
            assert npad_all <= 64 and p["drain_cols"] >= npad_all and not p["half"], where
            assert p["tmem_slots"] * p["drain_cols"] <= cols, where
        else:
            assert npad_all > 64, where
            per_buf = TMEM_COLS // p["tmem_buffers"]
            assert 1 <= p["tmem_slots"] <= 4 and p["tmem_slots"] <= p["kblocks"], where
            assert p["tmem_slots"] * p["npad"] <= per_buf or p["npad"] > 256, where
            # column halves only above 256 columns, on an even grid
            assert p["half"] == (npad_all > 256), where
            if p["half"]:
                assert p["grid"] % 2 == 0 and 2 * p["npad"] >= npad_all, where
                assert p["npad"] % 16 == 0 and p["npad"] <= 256, where
            else:
                assert p["npad"] == npad_all, where
        # at most one CTA per SM, no more CTAs than work
        ntile = -(-V // 128)
        assert 1 <= p["grid"] <= 152 and p["grid"] <= (2 * ntile if p["half"] else ntile), where
    assert n > 500


def test_contraction_plan_of_the_benchmark_shapes(lib):
    p = sv.spec_verify_plan(128256, 4096, 1, 4)
    assert (p["drain_cols"], p["chunks"], p["stages"], p["grid"]) == (16, 2, 6, 152)
    p = sv.spec_verify_plan(128256, 4096, 8, 7)
    assert p["drain_cols"] == 64 and p["tmem_slots"] == 8
    p = sv.spec_verify_plan(128256, 4096, 64, 5)
    assert p["half"] == 1 and p["npad"] == 192 and p["tmem_buffers"] == 2
    p = sv.spec_verify_plan(128256, 4096, 1, 4, "fp8")
    assert p["kblock_elems"] == 128 and p["kblocks"] == 32


def test_contraction_plan_rejects_what_create_rejects(lib):
    cfg = sv.sv_config_t(128256, 4096, 65, 5, sv.SV_BF16, None)   # 390 rows
    out = sv.sv_plan_t()
    assert lib.spec_verify_plan(ctypes.byref(cfg), 152, SMEM_OPTIN, ctypes.byref(out)) == \
        sv.SV_ERR_SHAPE
    cfg = sv.sv_config_t(128256, 4096, 1, 4, sv.SV_FP32, None)
    assert lib.spec_verify_plan(ctypes.byref(cfg), 152, SMEM_OPTIN, ctypes.byref(out)) == \
        sv.SV_ERR_ARG
    assert lib.spec_verify_plan(None, 152, SMEM_OPTIN, ctypes.byref(out)) == sv.SV_ERR_ARG
    # a GPU with too little shared memory for two stages
    cfg = sv.sv_config_t(128256, 4096, 1, 4, sv.SV_BF16, None)
    assert lib.spec_verify_plan(ctypes.byref(cfg), 152, 48 * 1024, ctypes.byref(out)) == \
        sv.SV_ERR_SHAPE


@pytest.mark.parametrize("path,shape,elt", [
    (bench.TRAFFIC_FILE, (128256, 4096, 1, 4), 2),
    (bench.TRAFFIC_FILE_B8K7, (128256, 4096, 8, 7), 2),
    (bench.TRAFFIC_FILE_FP8, (128256, 4096, 1, 4), 1),
])
def test_recorded_dram_traffic_is_one_pass_over_the_inputs(path, shape, elt):
    """A committed ncu figure that bench.py reports as `traffic` (only while
    its source hash matches the contraction's sources) reads the kernel's
    algorithmic bytes once: DRAM traffic within 1% above them (the rest is
    the logits and partials written back)."""
    traffic = bench.recorded_traffic(path)
    if traffic is None:
        pytest.skip("the contraction changed since this capture")
    algo = bench.contraction_bytes(*shape, elt=elt)
    assert algo <= traffic <= 1.01 * algo, (traffic, algo)
