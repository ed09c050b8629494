"""CPU checks of the benchmark's algorithmic-byte accounting against the
sizing figures the pages print."""
import bench


def test_kv_bytes_per_layer_llama7b_4096():
    """A LLaMA-7B layer (32 heads x 128, fp16/bf16) at 4096 tokens holds 64 MB
    of K and V (PD-disaggregation article, opening paragraph: 64 MB per layer,
    2 GB per token over 32 layers)."""
    kv = bench.masked_attend_bytes([4096], 32, 32, 4096, 128, 2)
    extra = 4096 + 2 * 32 * 128 * 2  # mask row, q and out
    assert kv - extra == 64 * 2**20
    assert 32 * (kv - extra) == 2 * 2**30


def test_copy_kvcache_volume():
    """Prefill -> generate copy of 32 layers x (K, V) x 32 heads x 1024 x 128
    x 2 bytes is 512 MB ("Intel NPU running LLMs", Part 5 '当前限制'); one
    append row moves read + write of that volume / 1024 per row."""
    per_row = bench.append_bytes(1, 32, 128, 2)  # read + write, K and V, one layer
    assert 32 * 1024 * per_row // 2 == 512 * 2**20


def test_paged_and_gather_accounting():
    lengths = [1, 128, 129]
    rows = sum(lengths)
    a = bench.paged_attend_bytes(lengths, 32, 8, 128, 2, 128)
    assert a == rows * 8 * 128 * 2 * 2 + (1 + 1 + 2) * 4 + 4 * 4 + 2 * 3 * 32 * 128 * 2
    g = bench.gather_bytes(lengths, 8, 128, 1, 64, 2, 128)
    assert g == 2 * rows * (8 * 128 + 64) * 2 + 4 * 4 + 4 * 4


def test_quantised_accounting_row_formats():
    """A quantised row is D E4M3 codes (one byte each), or D/2 bytes of E2M1
    code pairs, + one fp32 scale + 12 zero bytes: 144 or 80 bytes for
    D = 128, against 256 for a bf16 row, so the cache part of the attention
    bytes shrinks to 144/256 or 80/256 of the bf16 figure while the mask, q
    and out (bf16) stay."""
    lengths, Hq, Hkv, C, D = [1, 64, 700], 32, 8, 1024, 128
    rows = sum(lengths)
    assert bench.quant_row_bytes("gqa_fp8", D) == 144
    assert bench.quant_row_bytes("gqa_fp4", D) == 80
    b = bench.masked_attend_bytes(lengths, Hq, Hkv, C, D, 2)
    side = len(lengths) * C + 2 * len(lengths) * Hq * D * 2
    for row in (144, 80):
        f = bench.quant_attend_bytes(lengths, Hq, Hkv, C, D, row)
        assert f - side == rows * Hkv * 2 * row
        assert (f - side) * 256 == (b - side) * row
        # the append reads the bf16 row and writes the quantised one, K and V
        assert bench.quant_append_bytes(4, Hkv, D, row) == 4 * Hkv * 2 * (256 + row)


def test_paged_quantised_accounting():
    """The paged quantised step counts the valid quantised rows (144 or 80
    bytes), the table entries, the cumsum and the bf16 q and out: a bf16-row
    "quantised" row of 2 D bytes gives back the paged figure."""
    lengths, Hq, Hkv, D, BS = [1, 128, 129, 4000], 32, 8, 128, 128
    assert bench.paged_quant_attend_bytes(lengths, Hq, Hkv, D, 2 * D, BS) == \
        bench.paged_attend_bytes(lengths, Hq, Hkv, D, 2, BS)
    side = (1 + 1 + 2 + 32) * 4 + 5 * 4 + 2 * 4 * Hq * D * 2
    for row in (144, 80):
        assert bench.paged_quant_attend_bytes(lengths, Hq, Hkv, D, row, BS) == \
            sum(lengths) * Hkv * row * 2 + side
    assert bench.KV_FORMATS["paged_fp8"] == "E4M3" and bench.KV_FORMATS["gqa_fp4"] == "E2M1"


def test_indexed_accounting_counts_listed_rows_and_whole_lists():
    """Only the listed rows are read; every query's list is read whole
    (topk int32 entries, padding included)."""
    listed, topk, Hq, Hkv, D = [3, 2048, 0], 2048, 16, 1, 512
    a = bench.indexed_attend_bytes(listed, topk, Hq, Hkv, D, 2)
    assert a == (2051 * 1 * 512 * 2 * 2) + 3 * 2048 * 4 + 2 * 3 * 16 * 512 * 2
    # an empty list still reads its list, q and writes out
    assert bench.indexed_attend_bytes([0], topk, Hq, Hkv, D, 2) == 2048 * 4 + 2 * 16 * 512 * 2
