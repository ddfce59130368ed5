"""Layer roles and cache sharing of the 38-layer decode step, against the
layer lists and counts the pages give (host logic, no GPU).

Report reading ("把 KV Cache 压缩推到极限"), sections 三 (CED) and 四 (CSA2:
three modes): kv_source_layer_ids = [2, 8, 14, 20] are the Full layers that
produce main KV; index_source_layer_ids adds the four Reindex layers 24, 28,
32, 36; the other 30 of the 38 CSA2 layers are Reuse.  CSA2 page (SGLang
notes): a layer without its own compressor reads the main KV and index K of
the nearest preceding KV-source layer.  Q&A page ("DeepSeek-V4.1 模型结构（2）"):
each encoder Full layer adds half an entry per token (m = 2), the decoder's
one a whole entry (m = 1), 2.5 entries per token in all.
"""
from serving_lightning_indexer_gb300 import decode_step as ds

KV_SOURCE = [2, 8, 14, 20]
INDEX_SOURCE = [2, 8, 14, 20, 24, 28, 32, 36]


def test_roles_match_the_layer_lists():
    layers = list(ds.LAYERS)
    assert layers == list(range(2, 40))          # 38 CSA2 layers after the two SWA-only ones
    full = [l for l in layers if ds.role_of(l) == "full"]
    reindex = [l for l in layers if ds.role_of(l) == "reindex"]
    reuse = [l for l in layers if ds.role_of(l) == "reuse"]
    assert full == KV_SOURCE
    assert sorted(full + reindex) == INDEX_SOURCE
    assert len(reuse) == 30


def test_every_layer_reads_the_nearest_preceding_kv_source():
    for l in ds.LAYERS:
        src = max(s for s in KV_SOURCE if s <= l)
        assert ds.cache_of(l) == KV_SOURCE.index(src), l
    # the three encoder groups of six and the decoder's twenty layers
    assert [sum(1 for l in ds.LAYERS if ds.cache_of(l) == c) for c in range(4)] == [6, 6, 6, 20]


def test_compressed_entries_per_token():
    assert [ds.ratio_of(ds.cache_of(s)) for s in KV_SOURCE] == [2, 2, 2, 1]
    assert sum(1.0 / ds.ratio_of(ds.cache_of(s)) for s in KV_SOURCE) == 2.5


def test_keys_scored_per_step_of_the_benchmark_step():
    # batch 8 at {32K, 256K, 1M, 1M} x 2: three encoder Full layers score N/2
    # entries a sequence, the decoder Full layer N, four Reindex layers the
    # 2048 x 8 pool positions of each sequence
    lengths = [32768, 262144, 1 << 20, 1 << 20] * 2
    encoder = sum(n // 2 for n in lengths)
    decoder = sum(lengths)
    reindex = 8 * 2048 * 8
    assert ds.keys_scored(lengths) == 3 * encoder + decoder + 4 * reindex == 12_484_608
    # short sequences: the pool covers every entry
    assert ds.keys_scored([1000], layers=(24,)) == 1000
