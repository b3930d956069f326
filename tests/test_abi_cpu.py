"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, and its host logic (dispatch table, validation) behaves."""
import ctypes
import os
import re

import pytest

import synthetic_inputs as si
import transformer_linear_layer_gb300 as tll

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SM = 152


@pytest.fixture(scope="module", autouse=True)
def built():
    tll.build()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "lin.h")).read()
    return re.findall(r"LIN_API\s+[\w\s\*]+?\b(lin_\w+)\s*\(", src)


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("lin_create", "lin_forward", "lin_destroy", "lin_strerror"):
        assert required in names


def test_every_declared_symbol_is_exported():
    lib = ctypes.CDLL(tll.build())
    names = declared_functions()
    assert len(names) >= 10
    for name in names:
        assert hasattr(lib, name), f"{name} declared in lin.h but not exported"


def test_abi_version_and_messages():
    lib = tll.library()
    assert lib.lin_abi_version() == 1
    for code in (0, -1, -2, -3, -4, -5, -6):
        msg = lib.lin_strerror(code).decode()
        assert msg and msg != "unknown status"
    assert lib.lin_strerror(-99).decode() == "unknown status"


def test_null_context_is_an_argument_error():
    lib = tll.library()
    assert lib.lin_forward(None, 16, 16, 16, None, None, None, None, 0, 2, None) == tll.ERR_ARG
    assert lib.lin_check_device(None, None) == tll.ERR_ARG
    assert lib.lin_destroy(None) == tll.OK
    assert lib.lin_create(None, 0, 0) == tll.ERR_ARG
    # every other entry point that takes a context refuses a null one before touching a device
    assert lib.lin_forward_plan(None, None, 16, 16, 16, None, None, None, None, 0, 2, None) == tll.ERR_ARG
    assert lib.lin_forward_residual(None, 16, 16, 16, None, None, None, None, None, 0, 2, None) == tll.ERR_ARG
    assert lib.lin_backward_data(None, 16, 16, 16, None, None, None, 2, None) == tll.ERR_ARG
    assert lib.lin_backward_weight(None, 16, 16, 16, None, None, None, None, 2, None) == tll.ERR_ARG
    assert lib.lin_backward_data_gelu(None, 16, 16, 16, None, None, None, None, 2, None) == tll.ERR_ARG
    assert lib.lin_gelu_backward(None, 16, None, None, None, 2, None) == tll.ERR_ARG
    assert lib.lin_fold_layernorm(None, 16, 16, None, None, None, None, None, None, 0, None) == tll.ERR_ARG
    assert lib.lin_set_plan_override(None, 16, 16, 16, 2, 0, None) == tll.ERR_ARG
    assert lib.lin_clear_plan_overrides(None) == tll.ERR_ARG
    assert lib.lin_set_option(None, 1, 1) == tll.ERR_ARG
    assert lib.lin_attention_forward(None, 1, 128, 12, 64, None, None, None, 1, 0.0, None) == tll.ERR_ARG


def test_create_without_device_fails_cleanly():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p(123)
    assert tll.library().lin_create(ctypes.byref(h), 0, 0) == tll.ERR_CUDA
    assert not h.value


# ------------------------------------------------------------ dispatch table

def kname(p):
    return p.as_dict()["kernel_name"]


def test_dispatch_skinny_for_small_m_bf16():
    for M in (2, 5, 8, 16):  # (one row with X fitting in shared memory: the GEMV)
        p = tll.plan_query(SM, M, 4096, 4096, "bf16")
        assert kname(p) == "skinny" and p.splits > 1 and p.grid_y == p.splits
        assert p.grid_x * p.bn >= 4096 and p.grid_x * p.grid_y <= 2 * SM  # two CTAs per SM
    assert kname(tll.plan_query(SM, 17, 4096, 4096, "bf16")) == "tc"


def test_dispatch_tensor_cores_for_tf32_and_wide_bf16():
    for prec in ("tf32", "bf16"):
        p = tll.plan_query(SM, 8192, 50257, 768, prec)
        assert kname(p) == "tc"
        assert p.bn in (128, 192, 256) and p.grid_x == SM and p.grid_y == 1
        assert p.splits == 1 and p.workspace_bytes == 0
    small = tll.plan_query(SM, 200, 300, 64, "bf16")
    assert kname(small) == "tc" and small.grid_x == 2 * ((300 + small.bn - 1) // small.bn)


def test_dispatch_ffma_for_fp32():
    big = tll.plan_query(SM, 4096, 4096, 4096, "fp32")
    assert kname(big) == "ffma" and big.bm == 128 and big.splits == 1
    for N, K in ((2304, 768), (768, 768), (3072, 768), (768, 3072)):
        p = tll.plan_query(SM, 128, N, K, "fp32")
        assert kname(p) == "ffma" and p.bm == 64
        ctas = p.grid_x * p.grid_y * p.grid_z
        assert ctas >= SM // 2, (N, K, ctas)
        assert p.grid_z == p.splits


def test_dispatch_degenerate_shapes():
    assert kname(tll.plan_query(SM, 0, 10, 10, "bf16")) == "none"
    assert kname(tll.plan_query(SM, 10, 0, 10, "fp32")) == "none"
    assert kname(tll.plan_query(SM, 10, 10, 0, "tf32")) == "fill"
    with pytest.raises(tll.LinError):
        tll.plan_query(SM, -1, 10, 10, "bf16")
    with pytest.raises(tll.LinError):
        tll.plan_query(SM, 1, 10, 10, 9)


def test_split_respects_workspace():
    roomy = tll.plan_query(SM, 128, 768, 3072, "fp32", workspace_bytes=64 << 20)
    tight = tll.plan_query(SM, 128, 768, 3072, "fp32", workspace_bytes=2 << 20)
    none = tll.plan_query(SM, 128, 768, 3072, "fp32", workspace_bytes=0)
    assert roomy.splits > 1
    assert roomy.workspace_bytes <= 64 << 20 and tight.workspace_bytes <= 2 << 20
    assert tight.splits <= roomy.splits and none.splits == 1 and none.workspace_bytes == 0


def test_skinny_needs_no_workspace():
    p = tll.plan_query(SM, 16, 4096, 4096, "bf16", workspace_bytes=0)
    assert kname(p) == "skinny" and p.splits in (1, 2, 4, 8) and p.workspace_bytes == 0


def test_plan_make_families():
    for v in range(5):
        for s in (1, 2, 4, 8):
            p = tll.plan_make(SM, tll.KERNEL_SKINNY, v, s, 16, 4096, 4096, "bf16")
            assert p.splits == s and p.grid_y == s and p.grid_x == 32
    with pytest.raises(tll.LinError):
        tll.plan_make(SM, tll.KERNEL_SKINNY, 0, 3, 16, 4096, 4096, "bf16")
    with pytest.raises(tll.LinError):
        tll.plan_make(SM, tll.KERNEL_SKINNY, 5, 0, 16, 4096, 4096, "bf16")
    with pytest.raises(tll.LinError):
        tll.plan_make(SM, tll.KERNEL_SKINNY, 0, 0, 17, 4096, 4096, "bf16")
    with pytest.raises(tll.LinError):
        tll.plan_make(SM, tll.KERNEL_FFMA, 0, 0, 16, 64, 64, "bf16")
    for v, bn in ((0, 256), (1, 128), (2, 192), (3, 256), (4, 128), (5, 192)):
        p = tll.plan_make(SM, tll.KERNEL_TC, v, 2, 4096, 4096, 256, "tf32")
        assert p.bn == bn and p.grid_x == 2
    for width in (0, 1, 3, 151):
        p = tll.plan_make(SM, tll.KERNEL_TC, 3, width, 8192, 2304, 768, "bf16")
        assert p.grid_x % 2 == 0 and 2 <= p.grid_x <= SM
    with pytest.raises(tll.LinError):
        tll.plan_make(SM, tll.KERNEL_TC, 6, 0, 256, 256, 256, "tf32")
    p = tll.plan_make(SM, tll.KERNEL_FFMA, 1, 7, 128, 768, 768, "fp32")
    assert p.grid_z == 7 and p.workspace_bytes >= 7 * 128 * 768 * 4


def test_plan_make_stream_k():
    """TC stream-K plans: splits = 2, one workspace slot per CTA, single-CTA
    variants only, at least one tile per CTA; never the default."""
    p = tll.plan_make(SM, tll.KERNEL_TC, 0, -1, 8192, 768, 768, "bf16")
    assert p.splits == 2 and p.grid_x == SM
    assert p.workspace_bytes >= SM * 128 * 256 * 4
    p = tll.plan_make(SM, tll.KERNEL_TC, 2, -5, 384, 640, 768, "tf32")
    assert p.splits == 2 and p.grid_x == 5 and p.bn == 192
    with pytest.raises(tll.LinError):   # SM pair
        tll.plan_make(SM, tll.KERNEL_TC, 3, -1, 8192, 768, 768, "bf16")
    p = tll.plan_make(SM, tll.KERNEL_TC, 0, -10, 384, 640, 768, "bf16")
    assert p.splits == 2 and p.grid_x == 9      # no more CTAs than the 3 x 3 tiles
    for M, N, K in ((8192, 768, 768), (8192, 2304, 768), (8192, 3072, 768), (8192, 768, 3072)):
        assert tll.plan_query(SM, M, N, K, "bf16").splits == 1


def test_dispatch_gemv_for_few_fp32_rows():
    for prec in ("fp32", "tf32"):
        for M in (1, 2, 3, 8):
            p = tll.plan_query(SM, M, 50257, 768, prec)
            assert kname(p) == "gemv" and p.bm in (1, 2, 4, 8) and p.bm >= M and p.workspace_bytes == 0
    # X (rows x K fp32) must fit in shared memory; else the tiled kernels
    assert kname(tll.plan_query(SM, 8, 4096, 4096, "fp32")) == "ffma"
    assert kname(tll.plan_query(SM, 9, 4096, 768, "fp32")) == "ffma"
    # bf16: one row, at most one 128-row tile of W per SM
    assert kname(tll.plan_query(SM, 1, 4096, 4096, "bf16")) == "gemv"
    assert kname(tll.plan_query(SM, 1, 128 * SM, 768, "bf16")) == "gemv"
    assert kname(tll.plan_query(SM, 1, 128 * SM + 1, 768, "bf16")) == "skinny"
    for M in (2, 4, 5):
        assert kname(tll.plan_query(SM, M, 4096, 4096, "bf16")) == "skinny"
    assert kname(tll.plan_query(SM, 1, 4096, 32768, "bf16")) == "skinny"  # X does not fit as fp32
    p = tll.plan_make(SM, tll.KERNEL_GEMV, 0, 3, 5, 1000, 520, "fp32")
    assert p.grid_x == 3 and p.bm == 8
    with pytest.raises(tll.LinError):
        tll.plan_make(SM, tll.KERNEL_GEMV, 0, 0, 5, 1000, 520, "bf16")
    with pytest.raises(tll.LinError):
        tll.plan_make(SM, tll.KERNEL_GEMV, 0, 0, 9, 1000, 520, "fp32")


def test_autotune_menu():
    """The tuner's menu: valid plans only, no duplicates, each family that can
    run the shape, and the built-in choice among them for the common shapes."""
    from transformer_linear_layer_gb300 import autotune

    for (M, N, K, prec, fams) in [(8192, 2304, 768, "bf16", {tll.KERNEL_TC}),
                                  (8, 768, 768, "bf16", {tll.KERNEL_SKINNY, tll.KERNEL_TC}),
                                  (4, 768, 768, "bf16", {tll.KERNEL_SKINNY, tll.KERNEL_TC, tll.KERNEL_GEMV}),
                                  (128, 3072, 768, "fp32", {tll.KERNEL_FFMA}),
                                  (1, 50257, 768, "fp32", {tll.KERNEL_FFMA, tll.KERNEL_GEMV}),
                                  (4096, 4096, 4096, "tf32", {tll.KERNEL_TC})]:
        menu = autotune.candidates(152, M, N, K, prec, 64 << 20)
        keys = [autotune._plan_key(p) for p in menu]
        assert len(keys) == len(set(keys))
        assert {p.kernel for p in menu} == fams
        assert all(p.workspace_bytes <= 64 << 20 for p in menu)
        assert autotune._plan_key(tll.plan_query(152, M, N, K, prec, "none")) in keys
    # no workspace: no split plans
    assert all(p.workspace_bytes == 0 for p in autotune.candidates(152, 128, 3072, 768, "fp32", 0))


def test_roofline_floor():
    from transformer_linear_layer_gb300 import autotune

    # bf16 M=16: HBM-bound, the weight dominates
    t = autotune.roofline_floor_s(16, 4096, 4096, "bf16")
    assert abs(t - 2 * (16 * 4096 * 2 + 4096 * 4096) / 6783.1e9) < 1e-12
    # bf16 8192^3: compute-bound
    t = autotune.roofline_floor_s(8192, 8192, 8192, "bf16")
    assert abs(t - 2 * 8192 ** 3 / 1891.6e12) < 1e-12


def test_autotune_features_and_residual_fit():
    """The cost model's inputs on known plans, and the residual regression
    recovering coefficients planted in synthetic timings."""
    import math
    import random

    from transformer_linear_layer_gb300 import autotune

    # 8192 x 2304 bf16 on 128 x 256 tiles: 64 x 9 = 576 tiles on 152 SMs -> 4 waves, 576 / 608 busy
    p = tll.plan_make(152, tll.KERNEL_TC, 0, 0, 8192, 2304, 768, "bf16")
    f = autotune.features(152, 8192, 2304, 768, "bf16", p)
    assert f["family"] == "tc" and abs(f["fill"] - 576 / 608) < 1e-12 and f["tile_fill"] == 1.0
    # 128 x 768 fp32 on 64 x 64 tiles split 3: 72 units in 304 slots; 100 rows pad to 128
    p = tll.plan_make(152, tll.KERNEL_FFMA, 1, 3, 100, 768, 768, "fp32")
    f = autotune.features(152, 100, 768, 768, "fp32", p)
    assert f["split"] == 3 and abs(f["fill"] - 72 / 304) < 1e-12 and abs(f["tile_fill"] - 100 / 128) < 1e-12
    # the prior: an HBM-bound skinny layer costs its bytes at the copy peak, split or not (on-chip reduce)
    p1 = tll.plan_make(152, tll.KERNEL_SKINNY, 0, 4, 16, 4096, 4096, "bf16")
    t = autotune.predict_prior_s(16, 4096, 4096, "bf16", autotune.features(152, 16, 4096, 4096, "bf16", p1))
    assert abs(t - autotune.roofline_floor_s(16, 4096, 4096, "bf16")) < 1e-12

    m = autotune.ResidualModel(ridge=1e-9)
    rng = random.Random(3)
    for _ in range(80):
        f = {"fill": rng.uniform(0.05, 1), "tile_fill": rng.uniform(0.3, 1), "split": rng.choice([1, 2, 4, 8]),
             "family": rng.choice(["tc", "tc_pair", "skinny", "ffma", "gemv"]), "stream_k": rng.random() < 0.2}
        true = 0.2 - 0.7 * math.log(1 / f["fill"]) + 0.1 * math.log2(f["split"]) + (0.3 if f["stream_k"] else 0)
        m.add(f, 1e-5 * math.exp(true), 1e-5)
    # trusted only once a fit has been made on enough samples (pruning uses the fit)
    assert not autotune.ResidualModel().trusted and not m.trusted
    m.fit()
    assert m.trusted
    coef = {r["feature"]: r for r in m.report()}
    assert abs(coef["bias"]["coef"] - 0.2) < 1e-3 and abs(coef["log_idle_waves"]["coef"] + 0.7) < 1e-3
    assert abs(coef["log2_split"]["coef"] - 0.1) < 1e-3 and abs(coef["stream_k"]["coef"] - 0.3) < 1e-3
    assert coef["log_idle_waves"]["prior"] == "OVERprices" and coef["ffma"]["prior"] == "as priced"


def test_skinny_ring_for_many_row_tiles():
    """More 128-row tiles of W than SMs: the 6 x 1 ring (two CTAs per SM)
    without a split; otherwise the 5 x 1 ring split over a cluster."""
    p = tll.plan_query(SM, 8, 50257, 768, "bf16")
    assert kname(p) == "skinny" and p.variant == 1 and p.splits == 1
    p = tll.plan_query(SM, 16, 4096, 4096, "bf16")
    assert p.variant == 4 and p.splits == 8


def test_autotune_save_format(tmp_path):
    """The tuner's table on disk: one entry per tuned signature with a winner,
    every plan field kept, readable back into a Plan (host only)."""
    import json

    from transformer_linear_layer_gb300 import autotune

    p = tll.plan_make(SM, tll.KERNEL_FFMA, 1, 3, 128, 768, 768, "fp32")
    reports = [{"shape": [128, 768, 768], "precision": "fp32", "epilogue": "none", "winner": p.as_dict()},
               {"shape": [16, 4096, 4096], "precision": "bf16", "epilogue": "none", "winner": None}]
    path = tmp_path / "plans.json"
    autotune.save(reports, str(path))
    table = json.loads(path.read_text())
    assert len(table) == 1 and table[0]["shape"] == [128, 768, 768]
    back = autotune._plan_from_dict(table[0]["plan"])
    assert autotune._plan_key(back) == autotune._plan_key(p)


def test_header_is_plain_c_and_links(tmp_path):
    """include/lin.h compiles as C99 with warnings as errors, and a C program
    linked against the built library runs its host-only calls (no GPU)."""
    import shutil
    import subprocess

    import importlib

    B = importlib.import_module("transformer_linear_layer_gb300.build")

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = B.build()
    here = os.path.dirname(os.path.abspath(__file__))
    exe = str(tmp_path / "c_abi_host_calls")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", B.INCLUDE,
           os.path.join(here, "c_abi_host_calls.c"), lib, "-Wl,-rpath," + os.path.dirname(lib), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count("ok ") == 11


def test_no_cpu_fallback_in_the_binding():
    """Host tensors are refused by every compute entry point of the binding
    (nothing is computed on the CPU), and so are mismatched dtypes and shapes."""
    import torch

    x = torch.randn(4, 64)
    w = torch.randn(8, 64)
    for call in (lambda: tll.forward(x, w),
                 lambda: tll.forward_residual(x, w, torch.zeros(4, 8)),
                 lambda: tll.backward_data(torch.randn(4, 8), w),
                 lambda: tll.backward_weight(torch.randn(4, 8), x),
                 lambda: tll.backward_data_gelu(torch.randn(4, 8), w, x),
                 lambda: tll.gelu_backward(torch.randn(4, 8), torch.randn(4, 8)),
                 lambda: tll.fold_layernorm(w, torch.ones(64))):
        with pytest.raises((ValueError, TypeError)):
            call()
    with pytest.raises(TypeError):
        tll.forward(x.bfloat16(), w)  # bf16 X with fp32 W
    with pytest.raises((ValueError, TypeError)):
        tll.forward(x, torch.randn(8, 63))  # K mismatch


def test_static_scratch_rule_on_the_host():
    """lin_forward_fp32_static runs the dispatch table's split, refusing a
    shape whose split needs more than the fixed array. The split fills the
    SMs, so its scratch grows with the SM count and not with the shape: every
    GPT-2 and square fp32 shape fits on 152 SMs, and the refusal shape of the
    GPU test needs more than the array only on a much larger device. The
    binding's constant is the header's."""
    import re

    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "lin.h")).read()
    m = re.search(r"#define LIN_STATIC_SCRATCH_BYTES \((\d+)u << (\d+)\)", hdr)
    assert m and int(m.group(1)) << int(m.group(2)) == tll.STATIC_SCRATCH_BYTES
    for sm in (132, 148, 152, 160):
        for layer in list(si.GPT2_M128_FP32) + [si.SQUARE_256_FP32, si.SQUARE_4096_FP32]:
            p = tll.plan_query(sm, layer.M, layer.N, layer.K, "fp32", workspace_bytes=1 << 62)
            assert p.workspace_bytes <= tll.STATIC_SCRATCH_BYTES, (sm, layer.name)
    M, N, K = 64, 512, 8192
    assert tll.plan_query(152, M, N, K, "fp32", workspace_bytes=1 << 62).workspace_bytes <= tll.STATIC_SCRATCH_BYTES
    big = tll.plan_query(1024, M, N, K, "fp32", workspace_bytes=1 << 62)
    assert big.splits > 1 and big.workspace_bytes > tll.STATIC_SCRATCH_BYTES


def test_timeline_needs_the_timeline_build():
    """lin_timeline is exported by the library build but only the timeline
    build records stamps; arguments are checked first."""
    lib = tll.library()
    assert lib.lin_timeline(tll.KERNEL_TC, None, 0, 1) == tll.ERR_UNSUPPORTED
    assert lib.lin_timeline(tll.KERNEL_SKINNY, None, 0, 0) == tll.ERR_UNSUPPORTED
    assert lib.lin_timeline(tll.TIMELINE_ATTENTION, None, 0, 1) == tll.ERR_UNSUPPORTED
    assert lib.lin_timeline(tll.KERNEL_FFMA, None, 0, 1) == tll.ERR_ARG
    buf = ctypes.create_string_buffer(64)
    assert lib.lin_timeline(tll.KERNEL_TC, buf, 0, 0) == tll.ERR_ARG
    assert lib.lin_timeline(tll.KERNEL_TC, None, 64, 0) == tll.ERR_ARG
