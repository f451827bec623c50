"""The benchmark's algorithmic byte floors (the roofline numerators), checked
against counts written out by hand from the workloads' shapes (no GPU; the
weights are unallocated placeholders of the right sizes)."""
import types

import numpy as np

import bench
import synth


def _placeholder(w_shapes: dict) -> dict:
    return {n: np.empty(shp, dtype=dt) for n, (shp, dt) in w_shapes.items()}


def test_gemma_batch_one_floor():
    """Workload 1: 3 steps x (all weights + the views' readable KV + one embedding row).
    Weights: table 262144 x 5120, pre 1024 x 10240, post 5120 x 1024, per block q 4096 x 1024, o 1024 x 4096,
    gate / up 4096 x 1024, down 1024 x 4096 (bf16), gains fp32.  KV: the sliding view reads 1024 positions, the
    full view 8192, each x 4 KV heads x 256 x 2 bytes x (K, V)."""
    m = synth.ModelSpec(d_t=5120, d_a=1024, n_blocks=4, n_q_heads=16, head_dim=256, n_kv_heads=4, d_ff=4096,
                        vocab=262144, dtype="bf16", block_view=(0, 0, 0, 1))
    shapes = {"tok_embd": ((262144, 5120), np.uint16), "w_pre": ((1024, 10240), np.uint16),
              "w_post": ((5120, 1024), np.uint16), "norm_e": ((5120,), np.float32), "norm_h": ((5120,), np.float32),
              "final_norm": ((1024,), np.float32)}
    for i in range(4):
        shapes.update({f"blk{i}.w_q": ((4096, 1024), np.uint16), f"blk{i}.w_o": ((1024, 4096), np.uint16),
                       f"blk{i}.w_gate": ((4096, 1024), np.uint16), f"blk{i}.w_up": ((4096, 1024), np.uint16),
                       f"blk{i}.w_down": ((1024, 4096), np.uint16)})
        for g in ("attn_norm", "post_attn_norm", "pre_ffn_norm", "post_ffn_norm"):
            shapes[f"blk{i}.{g}"] = ((1024,), np.float32)
        shapes[f"blk{i}.q_norm"] = ((256,), np.float32)
    weights = _placeholder(shapes)
    w = types.SimpleNamespace(model=m, B=1, N=3, kv_len=np.array([8192], np.int32), weights=weights,
                              views=[dict(window=1024, sink=0), dict(window=0, sink=0)],
                              weight_bytes=lambda: sum(a.nbytes for a in weights.values()))
    wbytes = (262144 * 5120 + 1024 * 10240 + 5120 * 1024 + 4 * (3 * 4096 * 1024 + 2 * 1024 * 4096)) * 2 \
        + (2 * 5120 + 1024 + 4 * (4 * 1024 + 256)) * 4
    kv = (1024 + 8192) * 4 * 256 * 2 * 2
    assert bench.draft_bytes_per_launch(w) == 3 * (wbytes + kv + 5120 * 2)
    assert bench.draft_bytes_per_launch(w) == 8764372992   # the figure the design notes quote


def test_nextn_floor():
    """Workload 7: per draft step all weights + the drafter KV's rows [0, pos] + an embedding row; per catch-up
    iteration eh_proj and the key / value rows of w_qkv; per catch-up row its embedding row and fp32 hidden
    state; and the key / value rows the call writes (16 KB a row: 4 KV heads x 256 x bf16 x K, V)."""
    m = synth.NextnSpec(d=4096, n_q_heads=16, head_dim=256, n_kv_heads=4, d_ff=12288, vocab=248320, dtype="bf16")
    shapes = {"tok_embd": ((248320, 4096), np.uint16), "eh_proj": ((4096, 8192), np.uint16),
              "w_qkv": ((6144, 4096), np.uint16), "w_o": ((4096, 4096), np.uint16),
              "w_gate": ((12288, 4096), np.uint16), "w_up": ((12288, 4096), np.uint16),
              "w_down": ((4096, 12288), np.uint16)}
    for g in ("enorm", "hnorm", "head_norm", "attn_norm", "ffn_norm"):
        shapes[g] = ((4096,), np.float32)
    shapes["q_norm"] = shapes["k_norm"] = ((256,), np.float32)
    weights = _placeholder(shapes)
    w = types.SimpleNamespace(model=m, B=1, N=3, weights=weights, kv_len=np.array([4096], np.int32),
                              n_cu=np.array([2], np.int32))
    allw = sum(a.nbytes for a in weights.values())
    row = 4 * 256 * 2 * 2
    catch = 2 * (4096 * 8192 * 2 + 2 * 4 * 256 * 4096 * 2) + 2 * (4096 * 2 + 4096 * 4)
    steps = 3 * allw + sum((4096 + 2 + k + 1) * row + 4096 * 2 for k in range(3))
    assert bench.nextn_bytes_per_launch(w) == catch + steps + (2 + 3) * row
