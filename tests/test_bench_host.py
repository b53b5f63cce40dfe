"""Host-side logic of bench.py, CPU only: the rate formula against the pages'
printed table, the roofline peak arithmetic and the command line."""
import pytest

import bench
from golden_io import page_gflops


def test_flop_count_matches_page():
    # "Matrix Multiplication -- Naive to Tiled", section 03: 2.15 billion at N = 1024
    assert round(bench.flops(1024, 1024, 1024) / 1e9, 2) == 2.15
    # "From 306 ms to 86 ms": 16.8 million elements of C at N = 4096
    assert round(4096 * 4096 / 1e6, 1) == 16.8


@pytest.mark.parametrize("row", page_gflops(), ids=lambda r: f"N{r[0]}-{r[1]}ms")
def test_rate_formula_reproduces_page_table(row):
    n, ms, gflops, dec = row
    half = 0.5 * 10.0 ** -dec            # the printed time is rounded to `dec` decimals
    lo = bench.tflops(n, n, n, (ms + half) / 1e3) * 1e3
    hi = bench.tflops(n, n, n, (ms - half) / 1e3) * 1e3
    assert lo - 0.5 <= gflops <= hi + 0.5


def test_fp32_peak_arithmetic():
    assert abs(bench.fp32_ffma_peak() - 152 * 128 * 2 * 2.07e9 / 1e12) < 1e-9
    assert abs(bench.fp32_ffma_peak(1485.0) / bench.fp32_ffma_peak() - 1485 / 2070) < 1e-12


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "1"])


def test_mode_selection():
    # unknown modes are refused before any GPU work; the extra modes exist
    with pytest.raises(SystemExit):
        bench.main(["--modes", "fp32,fp8"])
    assert set(bench.EXTRA_MODES) <= set(bench.ALL_MODES)
    assert bench.ALL_MODES[:3] == bench.MODES == ("fp32", "tf32", "bf16")
    # every selectable mode has a stated nominal peak or the FFMA peak formula
    assert all(m in bench.NOMINAL_TFLOPS for m in bench.ALL_MODES if m != "fp32")


def test_e2e_input_sets():
    # FP32 and TF32 read the same float32 A and B: the default step copies
    # two input sets, float32 first because the FP32 product runs first
    assert bench.e2e_input_groups(bench.MODES) == ["f32", "bf16"]
    assert bench.e2e_input_groups(("bf16", "fp32")) == ["bf16", "f32"]
    assert bench.e2e_input_groups(bench.ALL_MODES) == ["f32", "bf16", "fp16"]
    assert bench.e2e_input_groups(("tf32", "fp32_via_bf16")) == ["f32"]
    # the end-to-end step runs FP32, the longest product, last
    assert bench.e2e_order(bench.MODES) == ("tf32", "bf16", "fp32")
    assert bench.e2e_order(bench.ALL_MODES)[-1] == "fp32"
    assert sorted(bench.e2e_order(bench.ALL_MODES)) == sorted(bench.ALL_MODES)
    assert bench.e2e_input_groups(bench.e2e_order(bench.MODES)) == ["f32", "bf16"]
    # 4096^2: 2 x 64 MiB float32 + 2 x 32 MiB bfloat16 in, 3 x 64 MiB out
    h2d, d2h = bench.e2e_bytes_per_step(bench.MODES, 4096)
    assert h2d == 201326592 and d2h == 201326592
    assert set(bench.E2E_GROUP_OF) == set(bench.ALL_MODES)
