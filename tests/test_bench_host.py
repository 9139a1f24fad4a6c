"""bench.py's host-side plumbing, without a GPU: the oracle split that the
CPU baseline and the reference arm time (its concatenated counter ranges must
equal one call over the whole range), and the reference arm's JSON line."""
import concurrent.futures as cf
import json
import os
import subprocess
import sys

import numpy as np
import pytest

from helpers import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402

U32 = 1 << 32


@pytest.mark.parametrize("name", ["u32", "u64_below_1000", "i64_range", "normal_f32", "normal_f64",
                                  "dropout_fwd_p0.5", "exponential_f32", "u8", "normal_f32_pairs"])
@pytest.mark.parametrize("first", [0, U32 - 1000])
def test_split_equals_one_call(orc, name, first):
    n = 4099  # ranges of unequal length; the second case wraps the counter
    call = bench.oracle_calls(orc, n)[name]
    whole = call(first, 0, n)
    with cf.ThreadPoolExecutor(max_workers=3) as pool:
        for parts in (1, 3, 7):
            split = bench.run_split(call, first, n, pool, parts)
            assert split.dtype == whole.dtype and split.tobytes() == whole.tobytes()


def test_oracle_calls_cover_every_fill(orc):
    assert set(bench.oracle_calls(orc, 16)) == {s.name for s in bench.fill_specs() + bench.next_specs()}


def test_only_selects_fills_of_the_step_and_beyond():
    assert [s.name for s in bench.selected_specs("u32,exponential_f32")] == ["u32", "exponential_f32"]
    with pytest.raises(SystemExit):
        bench.selected_specs("no_such_fill")


def test_reference_arm_prints_the_contract_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "1", "--ref-sample", "4096"], capture_output=True, text=True, env=env,
                         cwd=ROOT, timeout=300, check=True).stdout
    d = json.loads(out.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["unit"] == "GiB/s" and d["value"] > 0
    assert d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == bench.host_cores()
    assert d["e2e"] == {"value": d["value"], "unit": "GiB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_traffic_lookup_ignores_unknown_kernels():
    assert bench.ncu_traffic("no_such_kernel", "dropout.cu") is None
