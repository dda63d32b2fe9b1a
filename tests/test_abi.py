"""The C-ABI library builds, loads and exports every entry point that
include/lookahead.h declares (no GPU needed: nothing is called)."""
import ctypes
import os
import re

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"LA_API[^;(]*?\b(la_\w+)\s*\(", src))
    return names


def test_library_exports_every_declared_symbol():
    from helpers import build_lib
    path = build_lib()
    lib = ctypes.CDLL(path)
    declared = _declared()
    assert len(declared) >= 18
    for name in sorted(declared):
        assert hasattr(lib, name), name


def test_binding_covers_every_symbol():
    import lossless_lookahead_decoding_gb300 as LA
    assert set(LA.EXPORTS) == _declared()
    for name in LA.EXPORTS:
        assert callable(getattr(LA, name))


def test_product_path_does_not_reference_oracle():
    pkg = os.path.join(ROOT, "lossless_lookahead_decoding_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in src and "from oracle" not in src and "liboracle" not in src, fn


def test_workspace_bytes_is_host_only_and_checks_shapes():
    """la_workspace_bytes needs no GPU: it holds at least the bf16 KV cache
    (2 x L x d_kv x max_seq x 2 bytes, growing with max_seq at that rate) and
    returns 0 for a shape the library refuses."""
    import lossless_lookahead_decoding_gb300 as LA
    from helpers import build_lib
    build_lib()

    def desc(**kw):
        f = dict(n_layers=32, d_model=4096, n_heads=32, n_kv_heads=32, head_dim=128, ffn=11008,
                 vocab=32000, max_seq=804, rms_eps=1e-5, rope_theta=1e4, dtype=LA.LA_BF16,
                 emb=1, layer_w=1, final_norm=1, lm_head=1, stream=None)
        f.update(kw)
        return LA.la_model_desc(**f)

    kv = lambda m: 2 * 32 * 32 * 128 * m * 2
    ws = LA.la_workspace_bytes(desc(), 15, 5, 15)
    assert kv(804) <= ws < kv(804) + (1 << 30)
    assert LA.la_workspace_bytes(desc(max_seq=804 + 1024), 15, 5, 15) - ws >= kv(1024)
    assert LA.la_workspace_bytes(desc(dtype=LA.LA_FP32), 15, 5, 15) > ws  # fp32 cache and activations
    # the widest windows of 128 rows are accepted (LA_ATTN_TC's own limit is checked by la_create)
    assert LA.la_workspace_bytes(desc(), 31, 3, 31) > 0 and LA.la_workspace_bytes(desc(), 32, 2, 0) > 0
    for bad, wng in [(dict(head_dim=96), (15, 5, 15)), (dict(n_kv_heads=3), (15, 5, 15)),
                     (dict(d_model=4000), (15, 5, 15)), (dict(emb=None), (15, 5, 15)),
                     (dict(), (40, 5, 0)), (dict(), (4, 1, 4)), (dict(), (4, 9, 4)), (dict(), (-1, 5, 2))]:
        assert LA.la_workspace_bytes(desc(**bad), *wng) == 0, (bad, wng)


def test_every_declaration_cites_the_pages_or_says_there_is_none():
    """Each LA_API declaration is preceded by a comment that names the section
    of the method's summary page defining the call ("Pages: ...") or says the
    pages have no counterpart."""
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        src = open(os.path.join(ROOT, "include", fn)).read()
        prev_end, n = 0, 0
        for m in re.finditer(r"LA_API[^;(]*?\b(la_\w+)\s*\(", src):
            start = src.rfind("/*", prev_end, m.start())
            assert start >= 0, m.group(1)
            comment = src[start:m.start()]
            assert "Pages:" in comment or "No counterpart" in comment, m.group(1)
            prev_end = src.index(";", m.end()) + 1
            n += 1
        assert n == len(_declared()) or fn != "lookahead.h"


def test_batched_workspace_grows_by_one_sequence_block_per_sequence():
    """la_workspace_bytes_batch needs no GPU: batch 1 is la_workspace_bytes;
    each further sequence adds the same block, which holds at least that
    sequence's bf16 KV cache; batch x T > 128 rows is refused."""
    import lossless_lookahead_decoding_gb300 as LA
    from helpers import build_lib
    build_lib()
    d = LA.la_model_desc(n_layers=32, d_model=4096, n_heads=32, n_kv_heads=32, head_dim=128, ffn=11008,
                         vocab=32000, max_seq=804, rms_eps=1e-5, rope_theta=1e4, dtype=LA.LA_BF16,
                         emb=1, layer_w=1, final_norm=1, lm_head=1, stream=None)
    W, N, G = 7, 5, 7  # T = 57 rows: two sequences fit one 128-row pass
    one = LA.la_workspace_bytes(d, W, N, G)
    assert LA.la_workspace_bytes_batch(d, W, N, G, 1) == one
    two = LA.la_workspace_bytes_batch(d, W, N, G, 2)
    assert two - one >= 2 * 32 * 32 * 128 * 804 * 2
    assert LA.la_workspace_bytes_batch(d, W, N, G, 3) == 0      # 171 rows
    assert LA.la_workspace_bytes_batch(d, W, N, G, 0) == 0
    # greedy rows: one per sequence, up to 128 sequences
    g1, g2 = LA.la_workspace_bytes_batch(d, 0, 2, 0, 1), LA.la_workspace_bytes_batch(d, 0, 2, 0, 2)
    assert LA.la_workspace_bytes_batch(d, 0, 2, 0, 128) == g1 + 127 * (g2 - g1)
    assert LA.la_workspace_bytes_batch(d, 0, 2, 0, 129) == 0


def test_sampling_setters_refuse_a_null_context_on_the_host():
    """la_set_sampling, la_set_top_k and la_set_top_p check their context
    before anything else: a NULL context is LA_ERR_ARG with no GPU call."""
    import lossless_lookahead_decoding_gb300 as LA
    from helpers import build_lib
    build_lib()
    L = LA.lib()
    assert L.la_set_sampling(None, 0.7, 1) == LA.LA_ERR_ARG
    assert L.la_set_top_k(None, 5) == LA.LA_ERR_ARG
    for p in (0.5, 1.0, 0.0, float("nan")):
        assert L.la_set_top_p(None, p) == LA.LA_ERR_ARG
