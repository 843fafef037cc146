"""Host-side helpers of bench.py that run without a GPU."""
import bench


def test_peak_of_reads_numbers_and_value_objects_and_falls_back():
    assert bench.peak_of({"hbm_gbs": 6780}, "hbm_gbs") == 6780.0
    assert bench.peak_of({"hbm_gbs": "6780.5"}, "hbm_gbs") == 6780.5
    assert bench.peak_of({"hbm_gbs": {"value": 6700, "unit": "GB/s"}}, "hbm_gbs") == 6700.0
    for bad in (None, [], {}, {"hbm_gbs": None}, {"hbm_gbs": "n/a"}, {"hbm_gbs": 0}, {"hbm_gbs": {"unit": "GB/s"}},
                {"bf16_tflops": 1900}):
        assert bench.peak_of(bad, "hbm_gbs") is None


def test_rank_seeds_and_single_process_max():
    assert bench.rank_token_seed(1, 0) == 1 and bench.rank_token_seed(1, 1) != bench.rank_token_seed(1, 0)
    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25
