"""The bench's algorithmic bytes per launch (the numerator of every GB/s it
reports), restated here from the per-unit table with the oracle's size
helpers: with c = codes + scales of a message,
  qwZ quant / dequant     2 + c           per weight element
  reorder + quant         2 + c           per rank-bucket element
  hop 1                   c + c/G         per rank-bucket element
  final hop + Adam        S c + 26        per owned parameter
  ring step               2 + c / 2 + 2c / 2 + c + 4 (first / middle / last)
and the step totals quoted for the llama-layer bucket."""
import oracle
from synth import workloads as W

import bench


def msg(n, block, bits):
    return oracle.codes_bytes(n, bits) + 4 * oracle.num_blocks(n, block)


def test_llama_step():
    q, g = W.LLAMA.qwz, W.LLAMA.qgz
    lb = bench.launch_bytes(W.LLAMA)
    assert [n for n, _ in lb] == ["qwz_quant", "qwz_dequant", "qgz_reorder_quant", "qgz_final_hop"]
    m_w = q.nranks * msg(q.shard, q.block, q.bits)
    m_g = g.nd * msg(g.bucket, g.block, g.bits)
    assert lb[0][1] == lb[1][1] == 2 * q.nranks * q.shard + m_w == 608_706_560
    assert lb[2][1] == 2 * g.nd * g.bucket + m_g == 4_060_151_808
    assert lb[3][1] == m_g + 26 * g.bucket == 6_083_903_488
    assert sum(b for _, b in lb) == 11_361_468_416  # "11.36 GB moved per step"


def test_two_hop_step():
    g = W.TWO_HOP.qgz
    lb = dict(bench.launch_bytes(W.TWO_HOP))
    m1 = g.nd * msg(g.bucket, g.block, g.bits)
    m2 = g.nd * msg(g.nodes * g.slice_elems, g.block, g.bits)
    assert lb["qgz_reorder_quant"] == 2 * g.nd * g.bucket + m1
    assert lb["qgz_hop1"] == m1 + m2 == 2_491_416_576
    assert lb["qgz_final_hop"] == m2 + 26 * g.bucket


def test_modes():
    q, g = W.LLAMA.qwz, W.LLAMA.qgz
    nd, b = g.nd, g.bucket
    m_g = nd * msg(b, g.block, g.bits)
    # three micro-batches: two accumulations, then the accumulator quantizer
    lb = bench.launch_bytes(W.LLAMA, microbatches=3)
    acc = [x for n, x in lb if n == "grad_accumulate"]
    assert acc == [6 * nd * b, 10 * nd * b]
    assert dict(lb)["qgz_reorder_quant_acc"] == 6 * nd * b + m_g
    # Adam -> qwZ fused: no quantize launch, the final hop also writes the int8 message
    lb = bench.launch_bytes(W.LLAMA, fuse_qwz=True)
    assert [n for n, _ in lb] == ["qwz_dequant", "qgz_reorder_quant", "qgz_final_hop_qwz"]
    assert dict(lb)["qgz_final_hop_qwz"] == m_g + 26 * b + nd * msg(g.slice_elems, g.block, 8)
    # hpZ: the gather reads the whole message and writes the bf16 weights
    lb = dict(bench.launch_bytes(W.LLAMA, hpz=True))
    assert lb["hpz_gather"] == q.nranks * msg(q.shard, q.block, q.bits) + 2 * q.phi
    # 7B: 27 quantize calls, the last on the tail shard, and the standalone Adam
    q7 = W.SEVEN_B.qwz
    lb = bench.launch_bytes(W.SEVEN_B)
    quants = [x for n, x in lb if n == "qwz_quant"]
    assert len(quants) == q7.calls == 27
    assert quants[-1] == 2 * q7.tail_shard + msg(q7.tail_shard, q7.block, q7.bits)
    assert dict(lb)["shard_adam"] == 30 * W.SEVEN_B.standalone_adam


def test_ring_steps():
    g = W.TWO_HOP.qgz
    nd, L = g.nd, g.slice_elems
    m = msg(L, g.block, g.bits)
    steps = [x for n, x in bench.launch_bytes(W.TWO_HOP, ring=True) if n == "ring_step"]
    assert len(steps) == nd
    assert steps[0] == nd * (2 * L + m)
    assert all(x == nd * (2 * L + 2 * m) for x in steps[1:-1])
    assert steps[-1] == nd * (2 * L + m + 4 * L)
