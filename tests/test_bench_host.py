"""Host-side pieces of bench.py that need no GPU."""
import bench
from kv_cache_compression_c128_gb300 import inputs


def test_windows_overlap_tells_tiled_from_overlapping_windows():
    tiled = inputs.make_case(2, 2048, 128, seed=inputs.BASE_SEED + 1)
    assert not bench.windows_overlap(tiled)
    # 16 windows of 128 rows inside 1024-token requests must share rows
    general = inputs.make_case(2, 2048, 128, seed=inputs.BASE_SEED + 2, block_size=16,
                               boundaries_per_req=16)
    assert bench.windows_overlap(general)


def test_workload_config_is_the_workload_alone():
    case = inputs.make_case(2, 2048, 128, seed=inputs.BASE_SEED + 1)
    cfg = bench.workload_config(case)
    assert cfg == bench.workload_config(case)
    assert cfg["outputs"] == case.num_outputs == 16
    assert cfg["algorithmic_bytes_per_call"] == bench.bytes_for(case)
    assert not {"timing", "launch", "parallelism"} & set(cfg)
