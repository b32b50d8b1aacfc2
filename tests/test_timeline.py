"""The timeline analysis on synthetic stamps (CPU)."""
import numpy as np

from split_bf16_gemm_swap_gb300.timeline import analyse


def test_phases_of_a_regular_pipeline():
    # GEMM i starts from b_i = 10 us * i, the previous GEMM's last epilogue
    # end.  Half the CTAs finish their prologue 1 us before b_i (placed early),
    # half 2 us after it; first full stages 2.5 / 3.0 us after b_i, 6 us of
    # streaming, epilogue 1 us later, so the last epilogue ends at b_{i+1}.
    G, C = 12, 8
    T = np.zeros((G, C, 4))
    late = np.array([0.0] * (C // 2) + [1.0] * (C // 2))
    for i in range(G):
        b = 10_000.0 * i
        T[i, :, 0] = b - 1_000 + late * 3_000
        T[i, :, 1] = b + 2_500 + late * 500
        T[i, :, 2] = T[i, :, 1] + 6_000
        T[i, :, 3] = T[i, :, 2] + 1_000
    r = analyse(T, first=3, count=6)
    assert abs(r["period_us"] - 10.0) < 1e-9
    assert abs(r["stream_med"] - 6.0) < 1e-9
    assert abs(r["last_full_to_epilogue_end_med"] - 1.0) < 1e-9
    assert abs(r["first_full_med"] - 2.75) < 1e-9 and abs(r["first_full_max"] - 3.0) < 1e-9
    assert abs(r["epilogue_end_max"] - 10.0) < 1e-9
    assert abs(r["prologue_end_med"] - 0.5) < 1e-9
    assert r["placed_before_prev_end"] == C // 2
    assert r["ctas"] == C
