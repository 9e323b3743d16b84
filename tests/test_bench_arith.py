"""The roofline arithmetic of bench.py against values worked out by hand from
the workload shapes (no GPU): algorithmic bytes per token are q, k, v, o, g
and beta moved once; chunk-GEMM FLOPs per token and value head are
2 (3 C dk + 2 C dv + 3 dk dv), counted densely; a decode step also moves
every state in and out once."""
from __future__ import annotations

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from chunkwise_gated_delta_gdn_gb300 import synth  # noqa: E402


def view(name):
    c0 = synth.case(name)

    class W:
        pass

    w = W()
    for f in ("H", "HV", "dk", "dv", "chunk", "gate_mode", "scale"):
        setattr(w, f, getattr(c0, f))
    w.tokens = c0.tokens
    w.dtype_name = "bf16" if str(c0.dtype).endswith("bfloat16") else "f32"
    return c0, w


# bytes / token: fp32 H=HV=2 at 64: q, k 2*2*64*4 + v, o 2*2*64*4 + g, beta 2*(2*4) = 2064;
# bf16 H=16, HV=48 at 128: q, k 2*16*128*2 + v, o 2*48*128*2 + g, beta 2*48*4 = 33152;
# KDA bf16 H=HV=32 at 128: 16384 + 16384 + g 32*128*4 + beta 32*4 = 49280.
# FLOPs / token: HV * 2 * (3 C dk + 2 C dv + 3 dk dv):
# 2*2*(3*64*64 + 2*64*64 + 3*64*64) = 131072; 48*2*(3*64*128 + 2*64*128 + 3*128*128) = 8650752;
# 32*2*(3*32*128 + 2*32*128 + 3*128*128) = 4456448.
@pytest.mark.parametrize("name, bytes_per_token, flops_per_token", [
    ("gdn_fp32_t256", 2064, 131072),
    ("gdn_bf16_t4096", 33152, 8650752),
    ("gdn_bf16_t32768", 33152, 8650752),
    ("kda_bf16_b2_t8192", 49280, 4456448),
    ("gdn_varlen_t131072", 33152, 8650752),
])
def test_path_bytes_and_flops(name, bytes_per_token, flops_per_token):
    c0, w = view(name)
    assert bench.algorithmic_bytes(w) == bytes_per_token * c0.tokens
    assert bench.algorithmic_flops(w) == flops_per_token * c0.tokens


def test_bench_workload_totals():
    """32,768 tokens: 1.086 GB and 2.835e11 FLOPs; at the measured peaks
    (6777 GB/s, 1719 TF/s sustained) 160 us of HBM and 165 us of tensor time."""
    c0, w = view("gdn_bf16_t32768")
    assert bench.algorithmic_bytes(w) == 1_086_324_736
    assert bench.algorithmic_flops(w) == 283_467_841_536
    assert bench.algorithmic_bytes(w) / 6777e9 * 1e6 == pytest.approx(160.3, abs=0.1)
    assert bench.algorithmic_flops(w) / 1719e12 * 1e6 == pytest.approx(164.9, abs=0.1)


def test_prep_reads_only_its_inputs():
    # q, k (2*16*128*2) and g, beta (2*48*4) per token
    c0, w = view("gdn_bf16_t32768")
    assert bench.algorithmic_bytes(w, "prep") == (8192 + 384) * 32768


def test_decode_bytes():
    # 256 states of 48 x 128 x 128 fp32 read and written, plus per token
    # q, k (2*16*128*2), v, o (2*48*128*2), g and beta (48*2*4)
    c0 = synth.case("gdn_decode_bf16_b256")
    want = 2 * 256 * 48 * 128 * 128 * 4 + 256 * (8192 + 24576 + 384)
    assert bench.decode_bytes(c0) == want == 1_619_099_648


def test_whole_job_rate_and_metric_names():
    assert bench.whole_job_rate(32768, 1.0, 4) == pytest.approx(4 * 32768 / 1e-3)
    assert bench.metric_of(synth.case("gdn_decode_bf16_b256")) == bench.METRIC_DECODE
    assert bench.metric_of(synth.case("prepost_bf16_t32768")) == bench.METRIC_PREPOST
    assert bench.metric_of(synth.case("gdn_bf16_t32768")) == bench.METRIC


def test_kernel_own_bytes_of_the_split_design():
    """The scan of the 32k workload reads v (48*128*2 B/token), g and beta
    (2*48*4) and writes o (48*128*2), and reads back the prep's images: per
    chunk 48 value-head images of 32 KB and 16 [K_next; Q] images of 32 KB,
    512 chunks.  The prep reads q, k (2*16*128*2), g and beta and writes those
    images.  (ncu measured 1.87 and 1.33 GB of DRAM traffic for the two
    kernels.)"""
    c0, w = view("gdn_bf16_t32768")
    images = 512 * (48 + 16) * 32768
    assert images == 1_073_741_824
    assert bench.kernel_design_bytes(w, "scan", c0) == 32768 * (2 * 12288 + 384) + images
    assert bench.kernel_design_bytes(w, "prep", c0) == 32768 * (8192 + 384) + images
    # packed: chunks are counted per sequence (a ragged tail is a whole chunk)
    cv, wv = view("gdn_varlen_t131072")
    cu = [0, 100, 164, 131072 - 1, 131072, 131072, 131072, 131072, 131072]
    chunks = 2 + 1 + (131072 - 1 - 164 + 63) // 64 + 1
    assert bench.kernel_design_bytes(wv, "scan", cv, cu) == (
        131072 * (2 * 12288 + 384) + chunks * 64 * 32768)
    # KDA at chunk 32: per chunk and value head a 10 KB [P1; AqkT] image, a
    # 16 KB gated [Kg; Qg] image and 128 decays; 2 x 256 chunks, 32 value heads.
    # The scan reads v, writes o (32*128*2 B/token each) and reads beta (32*4);
    # the prep reads q, k (2*32*128*2), g (32*128*4) and beta.  (ncu measured
    # 0.70 and 0.95 GB.)
    ck, wk = view("kda_bf16_b2_t8192")
    images_k = 512 * 32 * (10240 + 16384 + 512)
    assert bench.kernel_design_bytes(wk, "scan", ck) == 16384 * (2 * 8192 + 128) + images_k
    assert bench.kernel_design_bytes(wk, "prep", ck) == 16384 * (16384 + 16384 + 128) + images_k
    # the fp32 path has no split-design figure
    cf, wf = view("gdn_fp32_t256")
    assert bench.kernel_design_bytes(wf, "scan", cf) is None
