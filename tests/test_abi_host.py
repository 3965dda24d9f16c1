"""Host-side tests of the C ABI: the library loads and exports every entry
point the header declares; configuration checks; the physical page pool,
per-sequence tables and error paths.  No GPU: device pointers are fake
aligned addresses that the host logic never dereferences."""
import ctypes
import os
import re

import pytest

import sparse_paged_decode_logical_gb300 as spd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_entry_points():
    src = open(os.path.join(ROOT, "include", "spd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spd_[a-z_]+)\s*\(", src)))


def test_library_exports_every_declared_entry_point():
    L = spd.lib()
    names = header_entry_points()
    assert "spd_kv_append" in names and "spd_sparse_decode_attention" in names
    for n in names:
        assert hasattr(L, n), n


def cfg(**kw):
    base = dict(num_q_heads=4, num_kv_heads=2, head_dim=64, dtype="f16",
                logical_page=16, physical_page=64, num_physical_pages=8,
                max_seqs=3, max_context=4096, streaming=[False, True], sink=16,
                window=256, token_budget=512, reuse_interval=4, free_list_seed=0)
    base.update(kw)
    return spd.make_config(**base)


def fake_buffers(sizes):
    addr, out = 1 << 40, {}
    for f in spd.BUFFER_FIELDS:
        if sizes[f]:
            out[f] = addr
            addr += (sizes[f] + 4095) // 4096 * 4096
    return out


def new_ctx(**kw):
    c = cfg(**kw)
    return c, spd.spd_create(c, fake_buffers(spd.spd_query_sizes(c)))


def test_sizes_follow_documented_layouts():
    c = cfg()
    z = spd.spd_query_sizes(c)
    # 8 pages x 1 dynamic head x 64 tokens x 64 dims x 2 bytes
    assert z["k_pool"] == z["v_pool"] == 8 * 1 * 64 * 64 * 2
    # R = 4 logical pages per physical page, min and max rows
    assert z["meta"] == 8 * 1 * 4 * 2 * 64 * 2
    # 3 sequences x 1 streaming head x (16 + 256) slots x 64 x 2
    assert z["stream_k"] == z["stream_v"] == 3 * 1 * 272 * 64 * 2
    assert z["page_table"] == 3 * 64 * 4          # ceil(4096 / 64) blocks
    assert z["selection"] == 3 * 1 * 32 * 4       # 512 / 16 pages kept
    assert z["scratch"] > 0


@pytest.mark.parametrize("bad", [
    dict(num_q_heads=6), dict(num_q_heads=12, num_kv_heads=4, streaming=None),
    dict(head_dim=96), dict(dtype=7), dict(logical_page=8),
    dict(physical_page=40), dict(physical_page=8192), dict(max_seqs=0),
    dict(max_context=0), dict(reuse_interval=0), dict(window=0),
    dict(num_physical_pages=0), dict(num_q_heads=48, num_kv_heads=3, streaming=None),
])
def test_invalid_configs_rejected(bad):
    with pytest.raises(spd.SpdError) as e:
        spd.spd_query_sizes(cfg(**bad))
    assert e.value.name == "SPD_ERR_INVALID_ARG"


def test_all_streaming_needs_no_pool():
    c = cfg(streaming=[True, True], num_physical_pages=0)
    z = spd.spd_query_sizes(c)
    assert z["k_pool"] == 0 and z["page_table"] == 0 and z["selection"] == 0


def test_misaligned_buffer_rejected():
    c = cfg()
    b = fake_buffers(spd.spd_query_sizes(c))
    b["meta"] += 16
    with pytest.raises(spd.SpdError):
        spd.spd_create(c, b)


def test_hierarchical_page_mapping_in_order():
    # "LServe long-sequence LLM serving system", section 2.2: physical pages
    # of 64 tokens hold logical pages of 16; a sequence of 200 tokens spans
    # ceil(200/64) = 4 physical pages, handed out in pool order
    _, ctx = new_ctx()
    s = spd.spd_seq_create(ctx)
    spd.spd_seq_reserve(ctx, s, 200)
    assert spd.spd_get_page_table(ctx, s) == [0, 1, 2, 3]
    assert spd.spd_free_pages(ctx) == 4
    spd.spd_seq_reserve(ctx, s, 56)      # 256 tokens still fit in 4 pages
    assert spd.spd_get_page_table(ctx, s) == [0, 1, 2, 3]
    spd.spd_destroy(ctx)


def test_seeded_free_list_is_a_reproducible_permutation():
    tables = []
    for _ in range(2):
        _, ctx = new_ctx(free_list_seed=1234)
        s = spd.spd_seq_create(ctx)
        spd.spd_seq_reserve(ctx, s, 8 * 64)
        tables.append(spd.spd_get_page_table(ctx, s))
        spd.spd_destroy(ctx)
    assert tables[0] == tables[1]
    assert sorted(tables[0]) == list(range(8)) and tables[0] != list(range(8))


def test_exhaustion_is_all_or_nothing():
    _, ctx = new_ctx()
    a, b = spd.spd_seq_create(ctx), spd.spd_seq_create(ctx)
    spd.spd_seq_reserve(ctx, a, 6 * 64)
    with pytest.raises(spd.SpdError) as e:
        spd.spd_seq_reserve(ctx, b, 3 * 64)
    assert e.value.name == "SPD_ERR_NO_PAGES"
    assert spd.spd_get_page_table(ctx, b) == [] and spd.spd_free_pages(ctx) == 2
    spd.spd_seq_reserve(ctx, b, 2 * 64)
    assert spd.spd_free_pages(ctx) == 0
    spd.spd_seq_free(ctx, a)
    assert spd.spd_free_pages(ctx) == 6
    spd.spd_seq_reserve(ctx, b, 6 * 64)   # room for 384 tokens: 2 -> 6 pages
    assert len(spd.spd_get_page_table(ctx, b)) == 6


def test_capacity_and_bad_sequences():
    _, ctx = new_ctx()
    s = spd.spd_seq_create(ctx)
    with pytest.raises(spd.SpdError) as e:
        spd.spd_seq_reserve(ctx, s, 4097)
    assert e.value.name == "SPD_ERR_CAPACITY"
    spd.spd_seq_free(ctx, s)
    with pytest.raises(spd.SpdError) as e:
        spd.spd_seq_free(ctx, s)
    assert e.value.name == "SPD_ERR_BAD_SEQ"
    for bad in (-1, 3, 99):
        with pytest.raises(spd.SpdError):
            spd.spd_seq_info(ctx, bad)
    ids = [spd.spd_seq_create(ctx) for _ in range(3)]
    assert sorted(ids) == [0, 1, 2]
    with pytest.raises(spd.SpdError) as e:
        spd.spd_seq_create(ctx)
    assert e.value.name == "SPD_ERR_CAPACITY"


def test_call_order_and_argument_errors_change_nothing():
    _, ctx = new_ctx()
    s = spd.spd_seq_create(ctx)
    fake = 1 << 41
    # select / attend on an empty sequence
    with pytest.raises(spd.SpdError) as e:
        spd.spd_select_pages(ctx, fake, [s])
    assert e.value.name == "SPD_ERR_STATE"
    with pytest.raises(spd.SpdError) as e:
        spd.spd_sparse_decode_attention(ctx, fake, [s], fake)
    assert e.value.name == "SPD_ERR_STATE"
    # duplicated or unknown ids, zero tokens, beyond max_context, pool too small
    for args in ([s, s], 1), ([s, 2], 1), ([s], 0), ([s], 5000), ([s], 9 * 64):
        with pytest.raises(spd.SpdError):
            spd.spd_kv_append(ctx, args[0], args[1], fake, fake)
    info = spd.spd_seq_info(ctx, s)
    assert info["length"] == 0 and spd.spd_free_pages(ctx) == 8


def test_append_without_usable_device_fails_cleanly():
    # fake pointers: the first GPU-side step (binding the buffers' device)
    # fails, and nothing in the host tables moves
    _, ctx = new_ctx()
    s = spd.spd_seq_create(ctx)
    with pytest.raises(spd.SpdError) as e:
        spd.spd_kv_append(ctx, [s], 100, 1 << 41, 1 << 41)
    assert e.value.name in ("SPD_ERR_CUDA", "SPD_ERR_INVALID_ARG")
    assert spd.spd_seq_info(ctx, s)["length"] == 0
    assert spd.spd_free_pages(ctx) == 8 and spd.spd_get_page_table(ctx, s) == []


def test_status_strings():
    L = spd.lib()
    for code in range(8):
        assert L.spd_status_string(code)


def test_fp8_storage_halves_the_kv_buffers():
    z16 = spd.spd_query_sizes(cfg(head_dim=128))
    z8 = spd.spd_query_sizes(cfg(head_dim=128, kv_fp8=True, k_scale=[0.5, 2.0],
                                 v_scale=[1.0, 0.25]))
    for f in ("k_pool", "v_pool", "meta", "stream_k", "stream_v"):
        assert z8[f] * 2 == z16[f], f
    assert z8["page_table"] == z16["page_table"] and z8["selection"] == z16["selection"]


@pytest.mark.parametrize("bad", [
    dict(kv_fp8=True),                                   # head_dim 64
    dict(head_dim=128, kv_fp8=True, k_scale=[0.0, 1.0]),
    dict(head_dim=128, kv_fp8=True, v_scale=[1.0, -2.0]),
    dict(head_dim=128, kv_fp8=True, k_scale=[float("inf"), 1.0]),
    dict(head_dim=128, kv_fp8=True, v_scale=[float("nan"), 1.0]),
])
def test_fp8_configs_checked(bad):
    with pytest.raises(spd.SpdError) as e:
        spd.spd_query_sizes(cfg(**bad))
    assert e.value.name == "SPD_ERR_INVALID_ARG"


def test_scales_are_ignored_without_fp8_storage():
    z = spd.spd_query_sizes(cfg(k_scale=[0.0, -1.0]))
    assert z["k_pool"] == 8 * 1 * 64 * 64 * 2


def test_page_mass_arguments_checked_before_any_work():
    _, ctx = new_ctx()
    s = spd.spd_seq_create(ctx)
    fake = 1 << 41
    # no selection yet, then bad output pointers / capacity: nothing moves
    with pytest.raises(spd.SpdError) as e:
        spd.spd_sparse_decode_attention_page_mass(ctx, fake, [s], fake, 0, 0, fake, fake, 4)
    assert e.value.name == "SPD_ERR_STATE"
    for args in ((fake, 0, fake, fake, 4), (0, 0, 0, fake, 4), (0, 0, fake, fake, 0),
                 (0, 0, fake + 2, fake, 4)):
        with pytest.raises(spd.SpdError) as e:
            spd.spd_sparse_decode_attention_page_mass(ctx, fake, [s], fake, *args)
        assert e.value.name == "SPD_ERR_INVALID_ARG", args
    assert spd.spd_seq_info(ctx, s)["step_counter"] == 0


def pcfg(**kw):
    base = dict(num_q_heads=8, num_kv_heads=2, head_dim=128, dtype=1, rank=16, block=64,
                token_budget=256, dense_below=32768)
    base.update(kw)
    return spd.spd_prefill_config(**base)


def prefill_sizes(c, L):
    kb, ws = ctypes.c_int(), ctypes.c_size_t()
    st = spd.lib().spd_prefill_sizes(ctypes.byref(c), L, ctypes.byref(kb), ctypes.byref(ws))
    return st, kb.value, ws.value


def test_prefill_sizes_dense_and_sparse():
    st, kb, ws = prefill_sizes(pcfg(), 1000)            # below 32K: dense, 16 blocks
    assert st == 0 and kb == 16 and ws > 0
    st, kb, _ = prefill_sizes(pcfg(dense_below=0), 1000)  # sparse: 256 / 64 blocks
    assert st == 0 and kb == 4
    st, kb, _ = prefill_sizes(pcfg(dense_below=0, token_budget=10 ** 6), 1000)
    assert st == 0 and kb == 16
    st, _, _ = prefill_sizes(pcfg(dense_below=0), 64 * 8192 + 1)
    assert spd.STATUS[st] == "SPD_ERR_CAPACITY"


@pytest.mark.parametrize("bad", [dict(block=32), dict(rank=0), dict(rank=65), dict(head_dim=96),
                                 dict(token_budget=63), dict(num_q_heads=6), dict(dtype=3),
                                 dict(dense_below=-1)])
def test_prefill_configs_checked(bad):
    st, _, _ = prefill_sizes(pcfg(**bad), 1000)
    assert spd.STATUS[st] == "SPD_ERR_INVALID_ARG"
    assert spd.STATUS[prefill_sizes(pcfg(), 0)[0]] == "SPD_ERR_INVALID_ARG"


def test_prefill_arguments_checked_before_any_work():
    c = pcfg()
    _, _, ws = prefill_sizes(c, 1000)
    L = spd.lib()
    a = 1 << 41
    run = lambda q, w, n: L.spd_prefill_block_sparse_attention(
        ctypes.byref(c), 1000, q, a, a, a, a, a, None, w, n, None)
    assert spd.STATUS[run(a + 8, a, ws)] == "SPD_ERR_INVALID_ARG"   # q not 16-byte aligned
    assert spd.STATUS[run(a, a + 16, ws)] == "SPD_ERR_INVALID_ARG"  # workspace not 256-aligned
    assert spd.STATUS[run(a, a, ws - 1)] == "SPD_ERR_CAPACITY"      # workspace too small


def test_prefill_binding_checks_tensors_before_the_library():
    torch = pytest.importorskip("torch")
    L, Hq, Hkv, d, r = 70, 4, 2, 64, 8
    q = torch.zeros((L, Hq, d), dtype=torch.bfloat16)
    k = torch.zeros((L, Hkv, d), dtype=torch.bfloat16)
    w = torch.zeros((Hkv, d, r), dtype=torch.float32)
    with pytest.raises(ValueError):   # k and v must share q's dtype
        spd.prefill_block_sparse_attention(q, k, k.half(), w, w)
    with pytest.raises(ValueError):   # k's shape must follow q's
        spd.prefill_block_sparse_attention(q, k[:-1], k, w, w)
    with pytest.raises(ValueError):   # projections are fp32 [Hkv][d][r]
        spd.prefill_block_sparse_attention(q, k, k, w.half(), w)
    with pytest.raises(ValueError):   # fp16 / bf16 only
        spd.prefill_block_sparse_attention(q.float(), k.float(), k.float(), w, w)
