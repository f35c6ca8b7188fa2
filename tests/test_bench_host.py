"""Host logic of bench.py: algorithmic work per workload, and the multi-rank
aggregation (max of times over ranks, world-size 2 on gloo, CPU only)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from head_attention_attn_gb300.inputs import WORKLOADS, Case, make_inputs


def test_causal_gqa_flops_count_only_causal_pairs():
    c = WORKLOADS["causal_gqa_bf16_4x32q8kv_4096x128"]
    # 4 * D * S(S+1)/2 * Hq * B
    assert bench.flops_of(c) == 4 * 128 * (4096 * 4097 // 2) * 32 * 4 == 549_890_031_616


def test_window_flops_count_band_pairs():
    c = WORKLOADS["window128_bf16_4x12x8192x64"]
    # every row sees |i - j| <= 64 clipped to [0, 8191]
    pairs = sum(min(8191, i + 64) - max(0, i - 64) + 1 for i in range(8192))
    assert pairs == 1_052_608
    assert bench.flops_of(c) == 4 * 64 * pairs * 12 * 4


def test_decode_bytes():
    c = WORKLOADS["decode_bf16_64x32q8kv_8192x128"]
    assert bench.bytes_of(c) == 2_148_532_224
    assert bench.flops_of(c) == 4 * 128 * 8192 * 32 * 64


def test_key_padding_flops_use_the_valid_lengths():
    c = WORKLOADS["bidir_keypad_bf16_8x12x512x64"]
    _, _, _, kl = make_inputs(c)
    assert bench.flops_of(c, kl) == 4 * 64 * 12 * 512 * int(kl.sum())


def test_visible_pairs_small_cases():
    c = Case("x", "bf16", B=1, Hq=1, Hkv=1, Lq=3, Lk=5, D=64, pos_offset=2, mask_mode=1)
    assert bench.visible_pairs(c) == 3 + 4 + 5
    c = Case("x", "bf16", B=1, Hq=1, Hkv=1, Lq=4, Lk=4, D=64, mask_mode=3, window=2)
    assert bench.visible_pairs(c) == 1 + 2 + 2 + 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    r, w, local = bench.dist_setup()
    assert (r, w, local) == (rank, world, rank)
    assert dist.get_backend() == "gloo"
    t = bench.max_over_ranks(0.5 + rank, w)
    s = bench.sum_over_ranks(1.0 + rank, w)
    bench.barrier(w)
    q.put((rank, t, s))
    dist.destroy_process_group()


def test_two_rank_aggregation_on_gloo():
    if torch.cuda.is_available():
        pytest.skip("gloo selection only applies without a GPU")
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    assert res == [(0, 1.5, 3.0), (1, 1.5, 3.0)]


def test_kernel_hash_follows_code_not_comments(tmp_path, monkeypatch):
    # the DRAM-traffic figure is keyed by this hash: a comment edit keeps it, a code edit in the
    # kernel, in the shared headers (kernels.h decides which key tiles a CTA visits) or in the
    # compile flags drops it
    import shutil
    from head_attention_attn_gb300 import build as _build
    src = os.path.join(bench.ROOT, "head_attention_attn_gb300", "csrc")
    dst = tmp_path / "head_attention_attn_gb300" / "csrc"
    dst.mkdir(parents=True)
    for name in ("prefill_tc.cu", "decode_tc.cu", "common.cuh", "kernels.h"):
        shutil.copy(os.path.join(src, name), dst / name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    assert h0 == bench.kernel_source_hash("prefill")
    assert h0 != bench.kernel_source_hash("decode_tc")
    with open(dst / "prefill_tc.cu", "a") as f:
        f.write("\n// a comment\n/* and a block\n   comment */\n\n")
    assert bench.kernel_source_hash() == h0
    with open(dst / "kernels.h", "a") as f:
        f.write("\nconstexpr int kUnusedInKernels = 1;\n")
    h1 = bench.kernel_source_hash()
    assert h1 != h0
    with open(dst / "common.cuh", "a") as f:
        f.write("\nconstexpr int kUnused = 1;\n")
    h2 = bench.kernel_source_hash()
    assert h2 != h1
    monkeypatch.setattr(_build, "NVCC_FLAGS", _build.NVCC_FLAGS + ["-DSOMETHING"])
    assert bench.kernel_source_hash() != h2


def test_paged_prefill_inputs_place_every_cached_position_once():
    """The timed chunked prefill's pools: every (sequence, page) entry names a distinct pool
    page, so every cached position of every sequence lives in exactly one pool row."""
    g = torch.Generator().manual_seed(3)
    for ps in (16, 128):
        q, out, cu, kv_lens, k_pool, v_pool, table = bench.paged_prefill_inputs(ps, "cpu", g)
        S = bench.PAGED_SHAPE
        B, chunk, kv = S["B"], S["chunk"], S["kv"]
        assert tuple(q.shape) == (B * chunk, S["Hq"], S["D"]) and out.shape == q.shape
        assert cu.tolist() == [chunk * b for b in range(B + 1)]
        assert kv_lens.tolist() == [kv] * B
        assert tuple(k_pool.shape) == (B * kv // ps, S["Hkv"], ps, S["D"]) and v_pool.shape == k_pool.shape
        assert tuple(table.shape) == (B, kv // ps)
        assert sorted(table.flatten().tolist()) == list(range(B * kv // ps))
