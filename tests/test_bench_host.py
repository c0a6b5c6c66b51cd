"""Host-side logic of the benchmark: the byte/flop model against the Muse Spark Open explainer's
own worked numbers (sections 10-14), and the multi-process (replica) timing path on CPU with
gloo ranks."""
import math
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def test_expert_size_model_matches_the_explainer():
    # section 10: one expert holds about 50 million weights (3 matrices of 4096 x 4096)
    d = I = 4096
    assert abs(3 * d * I / 1e6 - 50.3) < 0.1
    # section 11/13: at about 4.5 bits per weight one expert is about 28 MB ...
    b = bench.expert_bytes(d, I, bits_per_weight=4.5)
    assert abs(b / 1e6 - 28.3) < 0.1
    # ... read in about 5.9 us (an H200-class 4.8 TB/s), and about 21 us in bf16
    assert abs(bench.read_time_us(b, 4.8e12) - 5.9) < 0.05
    assert abs(bench.read_time_us(bench.expert_bytes(d, I, 16), 4.8e12) - 21.0) < 0.1
    # compute: 2 flops per weight per token, about 0.1 us per token at about 1 PFLOP/s
    f = bench.flops_per_token_expert(d, I)
    assert abs(f / 1e6 - 100.7) < 0.1
    t_tok = f / 1.0e15 * 1e6
    assert abs(t_tok - 0.1) < 0.001
    # crossover where reading and computing take equally long: about 58 tokens per expert
    assert 56 <= bench.crossover_tokens(5.9, 0.1) <= 60
    # section 12: 753 tokens x 8 choices over 256 experts is about 24 tokens per expert
    assert abs(753 * 8 / 256 - 23.5) < 0.1
    # section 14: 32 experts per GPU read once is about 190 us; 3,012 tokens x 8 / 8 GPUs of
    # compute at 0.1 us is about 300 us
    assert abs(32 * 5.9 - 189) < 1
    assert abs(3012 * 8 / 8 * 0.1 - 301) < 1


def test_mxfp4_bytes_per_weight():
    # 4 bits + one 8-bit scale per 32 weights = 4.25 bits; a decode-config expert is 26.7 MB
    assert bench.matrix_bytes(32, 32) == 32 * 32 * 4.25 / 8
    assert abs(bench.expert_bytes(8192, 2048) / 1e6 - 26.74) < 0.01
    lb = bench.layer_algorithmic_bytes(8192, 2048, 128, 1, 8)
    assert abs(lb / 1e6 - 218.1) < 0.2


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    r, w, lr = bench.dist_env()
    bench.init_dist(w, "gloo")
    bench.barrier(w)
    worst = bench.max_over_ranks(10.0 + r, w, "cpu")
    q.put((r, w, lr, worst))
    dist.destroy_process_group()


def test_replica_timing_takes_the_max_over_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    assert [r[0] for r in res] == [0, 1] and all(r[1] == 2 for r in res)
    assert all(r[3] == 11.0 for r in res)


def test_recorded_traffic_only_for_its_workload_and_sources():
    import bench
    src = ["bit_expert_ffn_moe_gb300/csrc/umma.cu", "bit_expert_ffn_moe_gb300/csrc/common.cuh"]
    assert bench.ncu_traffic("no_such_profile.md", src, "prefill") is None
    assert bench.ncu_traffic("umma_grouped_prefill.md", src, "long_prefill") is None
    assert bench.ncu_traffic("umma_grouped_prefill.md", src[:1], "prefill") is None  # other sources


def test_traffic_only_for_the_plain_launch():
    """A launch at the latent width, or the decode kernel on MXFP8 activations, matches no summary
    (all were captured on the plain layer)."""
    import argparse

    import bench
    from bit_expert_ffn_moe_gb300 import inputs as IN
    cfg = IN.CONFIGS["decode"]
    assert bench.traffic_workload(argparse.Namespace(latent=0), cfg) == "decode"
    assert bench.traffic_workload(argparse.Namespace(latent=4096), cfg) == "decode+latent4096"
    assert bench.traffic_workload(argparse.Namespace(latent=0), cfg, "+mxfp8") == "decode+mxfp8"
    assert bench.ncu_traffic("umma_decode_layer.md", bench.DECODE_KERNEL_SOURCES, "decode+mxfp8") is None


def test_variant_options_name_the_workload_and_count_launches():
    """--expert-norm and --latent change the layer the bench times: the workload name says so,
    the layer runs at the latent width, and the launch count includes the extra kernels."""
    import argparse

    from bit_expert_ffn_moe_gb300 import inputs as IN
    cfg = IN.CONFIGS["decode"]
    plain = argparse.Namespace(expert_norm=False, latent=0)
    both = argparse.Namespace(expert_norm=True, latent=4096)
    assert bench.workload_name(plain, cfg) == cfg.note
    name = bench.workload_name(both, cfg)
    assert "8192 -> 4096 -> 8192" in name and "RMSNorm" in name
    assert bench.moe_cfg(plain, cfg) is cfg
    cm = bench.moe_cfg(both, cfg)
    assert (cm.d, cm.E, cm.k, cm.I, cm.T) == (4096, cfg.E, cfg.k, cfg.I, cfg.T)
    assert bench.norm_eps(plain) is None and bench.norm_eps(both) == 1e-6
    # decode: fused router, gate/up, down+sum; + the normalising sum; + 2 x (plan + GEMV)
    assert bench.launches_per_step(0, 1, 8192, 128, 8) == 3
    assert bench.launches_per_step(0, 1, 8192, 128, 8, expert_norm=True) == 4
    assert bench.launches_per_step(0, 1, 8192, 128, 8, latent=True) == 7
    # prefill: 7 layer kernels (logits, counting top-k, permutation, operand rows, up, down, sum);
    # + 2 x (plan, operand rows, GEMM)
    # tensor-core decode: route, token pieces, the fused expert kernel (its sum fused up to 4 tokens)
    # up to eight tokens: the expert kernel routes its own tokens (one launch; + the normalising sum)
    assert bench.launches_per_step(1, 4096, 8192, 128, 8) == 10          # screened router: + 3
    assert bench.launches_per_step(1, 200, 8192, 128, 8) == 7            # dense router below 256 tokens
    assert bench.launches_per_step(1, 65536, 8192, 1024, 8) == 7         # and beyond 2^25 token-expert pairs
    assert bench.launches_per_step(0, 1, 8192, 128, 8, mma_decode=True) == 1
    assert bench.launches_per_step(0, 4, 8192, 128, 8, mma_decode=True) == 1
    assert bench.launches_per_step(0, 8, 8192, 128, 8, mma_decode=True) == 2
    assert bench.launches_per_step(0, 16, 8192, 128, 8, mma_decode=True) == 6   # logits, top-k, permutation,
    assert bench.launches_per_step(0, 8, 8192, 200, 8, mma_decode=True) == 4    # pieces, experts, sum
    assert bench.launches_per_step(0, 16, 8192, 128, 8) == 5                     # BF16 GEMVs beyond 8 tokens
    assert bench.launches_per_step(0, 1, 8192, 128, 8, expert_norm=True, mma_decode=True) == 2
    assert bench.launches_per_step(1, 4096, 8192, 128, 8) == 10
    assert bench.launches_per_step(1, 4096, 8192, 128, 8, latent=True) == 16


def test_nvfp4_weight_option_changes_the_byte_model_and_the_names():
    """--weights nvfp4: 4.5 bits per weight (one E4M3 byte per 16 values) plus a 4-byte global
    scale per matrix; the workload and dtype name the format."""
    import argparse

    from bit_expert_ffn_moe_gb300 import inputs as IN
    cfg = IN.CONFIGS["decode"]
    d, I = cfg.d, cfg.I
    assert bench.expert_read_bytes(d, I) == bench.expert_bytes(d, I) == 3 * (I * d // 2 + I * d // 32)
    assert bench.expert_read_bytes(d, I, "nvfp4") == 3 * (I * d // 2 + I * d // 16 + 4)
    assert bench.up_bytes_per_expert(d, I, "nvfp4") == 2 * (I * d // 2 + I * d // 16 + 4)
    mx = bench.layer_algorithmic_bytes(d, I, cfg.E, 1, 8)
    nv = bench.layer_algorithmic_bytes(d, I, cfg.E, 1, 8, "nvfp4")
    assert nv - mx == 8 * 3 * (I * d // 32 + 4)
    args = argparse.Namespace(expert_norm=False, latent=0, weights="nvfp4")
    assert "NVFP4" in bench.workload_name(args, cfg)
    assert bench.dtype_name(0, "nvfp4").startswith("nvfp4 weights x bf16")


def test_parity_gate_accepts_the_oracle_and_refuses_a_wrong_output():
    import numpy as np
    rng = np.random.default_rng(0)
    ys = [rng.standard_normal((1, 64)).astype(np.float32) for _ in range(3)]
    res = bench.parity_gate(ys, ys)
    assert res["ok"] and res["rows_checked"] == 3 and res["rel_fro"] == 0.0
    bad = [y.copy() for y in ys]
    bad[1][0, 5] += 1.0  # one wrong element
    with pytest.raises(RuntimeError, match="refusing to record"):
        bench.parity_gate(bad, ys)
    with pytest.raises(RuntimeError, match="refusing to record"):
        bench.parity_gate([np.zeros((1, 64))] * 3, ys)  # an all-zero output
    with pytest.raises(RuntimeError, match="refusing to record"):
        bench.parity_gate(ys[:2], ys)


@pytest.mark.parametrize("T,weights,norm", [(2, "mxfp4", False), (16, "mxfp4", True), (2, "nvfp4", False)])
def test_oracle_sample_outputs_are_the_parity_rows(T, weights, norm):
    """The oracle sample returns, row for row, the outputs of the inputs parity_inputs() names,
    computed with the sampled layer copy's weights; threads=1 runs on one thread."""
    import argparse

    import numpy as np

    from bit_expert_ffn_moe_gb300 import inputs as IN
    from oracle import oracle as O
    cfg = IN.small_config("sample_T%d" % T, T=T, d=256, E=8, k=2, I=256, index=150 + T)
    args = argparse.Namespace(fmt="bf16", weights=weights, latent=0, expert_norm=norm, layers=4)
    res = bench.oracle_sample(args, cfg, 3, threads=1)
    assert res["cores"] == 1
    inputs = bench.parity_inputs(cfg, 3)
    li = bench.sample_layer_index(args)
    assert li == 1
    W_r, b = IN.make_router(cfg)
    W_r = (np.random.default_rng([cfg.seed, 77, li]).standard_normal(W_r.shape) / np.sqrt(cfg.d)).astype(np.float32)
    pack = O.nvfp4_pack if weights == "nvfp4" else O.mxfp4_pack

    def wts(e):
        return {n: pack(IN.synth_weights(cfg.seed + 7919 * li, t, e, *IN.expert_matrix_shapes(cfg)[t], cfg.weight_std))
                for n, t in (("gate", IN.TENSOR_GATE), ("up", IN.TENSOR_UP), ("down", IN.TENSOR_DOWN))}
    assert len(res["ys"]) == len(inputs)
    for (xb, rows), y in zip(inputs, res["ys"]):
        ref = O.moe_layer(xb, W_r, b, cfg.k, wts, O.ACT_BF16,
                          expert_norm_eps=bench.EXPERT_NORM_EPS if norm else None)["y"]
        np.testing.assert_array_equal(y, ref if rows is None else ref[rows])
    assert O.max_threads() == len(__import__("os").sched_getaffinity(0))  # restored


def test_default_line_times_verify_and_the_prefill_workloads_in_both_activation_formats():
    import argparse
    a = argparse.Namespace(extra="auto", config="decode", latent=0, expert_norm=False, weights="mxfp4", fmt="bf16")
    names = bench.extra_workloads(a)
    assert names == ["spec_verify", "prefill", "long_prefill", "prefill_mxfp8"]
    assert [bench.EXTRA_WORKLOADS[n] for n in names] == [("spec_verify", "bf16"), ("prefill", "mxfp4"),
                                                          ("long_prefill", "mxfp4"), ("prefill", "mxfp8")]
    a.fmt = "mxfp8"  # a variant headline times nothing else
    assert bench.extra_workloads(a) == []
    # the prefill roofline is the FP4 tensor peak for MXFP4 activations, FP8 for MXFP8 beyond 16
    # tokens; MXFP8 up to 16 tokens runs the decode kernels (HBM-bound)
    assert bench.grouped_gemm_path(1, 1) and bench.grouped_gemm_path(2, 17) and not bench.grouped_gemm_path(2, 16)
    assert bench.tensor_peak_ratio(1) == 6.0 and bench.tensor_peak_ratio(2) == 2.0
    assert bench.launches_per_step(2, 1, 8192, 128, 8, mma_decode=True) == bench.launches_per_step(
        0, 1, 8192, 128, 8, mma_decode=True)
    assert bench.launches_per_step(2, 4096, 8192, 128, 8) == 10
