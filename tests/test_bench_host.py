"""Host-side arithmetic of bench.py (no GPU): stage partition, the gate/up launches' algorithmic
bytes that the roofline divides by their durations, and the source hash that ties the ncu
traffic figure to the kernel it was taken with."""
import json
import os

import bench
import spd_inputs as si


def test_stage_sizes_follow_the_floor_bounds():
    # b_s = floor(s L / n): 36 layers over 8 stages alternate 4 and 5
    assert bench.stage_sizes(36, 8) == [4, 5, 4, 5, 4, 5, 4, 5]
    assert bench.stage_sizes(5, 4) == [1, 1, 1, 2]
    assert sum(bench.stage_sizes(28, 3)) == 28


def test_gateup_bytes_count_occupied_stages_per_round():
    dm = si.SHAPE_4B.dims
    per = 2 * dm.F * dm.d * 2
    # a full pipeline: rounds 0..3 have all 8 stages, round 4 only the 5-layer stages
    full = [{"n_active": 8}]
    b, launches = bench.gateup_bytes(full, dm, 8)
    assert launches == 5
    assert b == per * (8 * 4 + 4)
    # right after a flush only stage 0 is occupied: one stage-layer per round it has a layer
    b1, l1 = bench.gateup_bytes([{"n_active": 1}], dm, 8)
    assert l1 == 5 and b1 == per * 4


def test_traffic_file_is_a_per_stage_layer_figure():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "profiles", "gateup_traffic.json")) as f:
        tj = json.load(f)
    src = os.path.join(root, "speculative_pipeline_decoding_spd_gb300", "csrc", "k_target.cu")
    # the figure is tied to one source (bench.py reports traffic null for any other)
    assert len(bench.source_hash(src)) == 16 and len(tj["k_target_sha"]) == 16
    # DRAM bytes of one stage-layer of gate/up: its weights once, plus the small outputs
    alg = 2 * si.SHAPE_4B.dims.F * si.SHAPE_4B.dims.d * 2
    assert alg * 0.99 < tj["dram_bytes_per_stage_layer"] < alg * 1.05


def test_alpha_ref_is_the_closed_form_or_one_over_n():
    assert bench.alpha_ref("forced-0.6", 8) == 1.0 / (1.0 + 7 * 0.4)
    assert bench.alpha_ref("forced-1.0", 8) == 1.0
    assert bench.alpha_ref("greedy", 8) == 1.0 / 8
    assert bench.alpha_ref("t1", 8) is None
    assert bench.cpu_alpha("t1", 8, 0.31) == 0.31
    assert bench.cpu_alpha("forced-0.3", 8, 0.5) == 1.0 / (1.0 + 7 * 0.7)


def test_workload_selection():
    class A:
        mode, shape, n = "forced-0.6", "4b", 0
    assert bench.select_workload(A) is si.SHAPE_4B
    A.mode = "t1"
    assert bench.select_workload(A) is si.SHAPE_4B_T1
    A.mode, A.shape, A.n = "forced-0.7", "8b", 16
    wl = bench.select_workload(A)
    assert wl.dims == si.SHAPE_8B.dims and wl.n == 16 and wl.prompt_len == 4096 and wl.Ls == 2


def test_l2_note_follows_the_bytes_streamed_per_step():
    # the 4B workload streams gigabytes per step: no flush; the tiny fp32 model sits in L2
    assert bench.l2_note(6.1e9).startswith("no flush needed")
    assert bench.l2_note(23e6).startswith("L2-resident")
