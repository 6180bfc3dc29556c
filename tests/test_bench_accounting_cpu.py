"""The benchmark's algorithmic accounting (the numerator of every roofline
figure) against closed forms written out from each workload's sizes: bytes
of cache a decode call must read, plus its queries, outputs and appended
rows, and the latent call's multiply-add work."""
import bench
from kv_cache_decode_gqa_gb300 import workloads as W


def test_llama2_7b_bytes():
    s = W.config("llama2_7b_mha")
    per_token = 32 * 2 * 128 * 2          # kv heads x (K, V) x d x bf16
    assert bench.kv_bytes_layer(s) == 4097 * per_token == 67_125_248
    assert bench.kv_bytes_step(s) == 32 * 67_125_248
    # the fused call also reads q, writes out, and reads + writes the new row
    q = out = 32 * 128 * 2
    append = 2 * 32 * 128 * (2 + 2)
    assert bench.decode_launch_bytes(s) == 67_125_248 + q + out + append


def test_llama31_70b_bytes_and_fp8_half():
    s = W.config("llama31_70b_gqa")
    assert bench.kv_bytes_layer(s) == sum(s.seq_lens) * 8 * 2 * 128 * 2
    f = W.config("llama31_70b_gqa_fp8")
    assert f.seq_lens == s.seq_lens
    assert 2 * bench.kv_bytes_layer(f) == bench.kv_bytes_layer(s)


def test_sliding_window_reads_only_the_window():
    s = W.config("llama31_70b_gqa_fp8_swa")
    assert min(s.seq_lens) > 128
    assert bench.kv_bytes_layer(s) == 32 * 128 * 8 * 2 * 128 * 1


def test_mxfp4_row_is_72_bytes():
    s = W.config("llama2_7b_mha_mxfp4")
    # 64 bytes of 4-bit codes + 8 one-byte scales per 128-channel row
    assert bench.kv_bytes_layer(s) == 4097 * 32 * 2 * (64 + 8)


def test_mla_bytes_and_flops():
    s = W.config("mla")
    rows = 64 * 32_769
    assert bench.kv_bytes_layer(s) == rows * 576 * 2 == 2_415_992_832
    useful, issued = bench.latent_flops(s)
    # per head and cached row: 576 score and 512 value multiply-adds
    assert useful == 2 * rows * 128 * (576 + 512) == 584_133_378_048
    # the tensor-core kernel's two value halves each recompute the scores
    assert bench.LATENT_TC_PARTS == 2
    assert issued == 2 * rows * 128 * (2 * 576 + 512)


def test_sparse_schedule_bytes():
    s = W.config("sparse")
    gather = 8 * 2048 * 2 * 512 * 2       # selected K and V rows
    indexer = 8 * 131_073 * 64 * 2        # every visible indexer key
    assert gather == 33_554_432 and indexer == 134_218_752
    for layer, mode in enumerate(s.modes):
        want = gather + (indexer if mode in ("full", "reindex") else 0)
        assert bench.kv_bytes_layer(s, layer) == want, (layer, mode)


def test_data_description_names_the_cache_format():
    assert "bf16 cache" in bench.data_description(W.config("llama2_7b_mha"))
    assert "E4M3" in bench.data_description(W.config("llama31_70b_gqa_fp8"))
    assert "E2M1" in bench.data_description(W.config("llama2_7b_mha_mxfp4"))
    assert "bf16 cache" in bench.data_description(W.config("sparse"))


def test_latent_parts_match_the_library():
    # the issued-work accounting follows the kernel's value split
    import os
    import re
    h = os.path.join(os.path.dirname(__file__), "..", "kv_cache_decode_gqa_gb300",
                     "csrc", "kvd_internal.h")
    m = re.search(r"constexpr int kLatentTcParts = (\d+);", open(h).read())
    assert m and int(m.group(1)) == bench.LATENT_TC_PARTS
