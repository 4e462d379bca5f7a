"""GPU parity: the CUDA decode step (through the C ABI) against the CPU oracle on the same seeded
inputs.  Small workloads are compared token by token in full; the full-size workloads (the
configurations bench.py times, same launch configuration) on sampled sequences."""
import numpy as np
import pytest
import torch

import dsv4_inputs as I
from oracle import compare as CMP
from oracle import dsv4_oracle as O

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import deepseek_v4_hybrid_gb300 as M
    return M


def to_host(t):
    if t is None:
        return None
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def gpu_results(ds):
    g = {"swa_cache": to_host(ds.swa_cache), "out": to_host(ds.out), "lse": to_host(ds.lse)}
    if g["out"].dtype == np.uint16:
        g["out"] = O.bf16_decode(g["out"])
    if ds.q_prep:
        g["q_out"] = to_host(ds.q)
    if ds.has_compress:
        g["state"] = to_host(ds.state)
        g["main_cache"] = to_host(ds.main_cache)
    if ds.has_indexer:
        g["idx_cache"] = to_host(ds.idx_cache)
        g["topk_idx"] = to_host(ds.topk_idx)
        g["topk_score"] = to_host(ds.topk_score)
        if ds.cand_blocks is not None and ds.cand_write:
            g["cand_out"] = to_host(ds.cand_blocks)
    return g


def run_and_compare(name, seqs=None, given=False):
    from deepseek_v4_hybrid_gb300.step import DeviceStep
    cfg = I.ALL_CONFIGS[name]
    st = I.make_step(cfg)
    ds = DeviceStep(st, topk_override=st.given_topk if given else None)
    ds.run()
    torch.cuda.synchronize()
    import deepseek_v4_hybrid_gb300 as M
    assert M.dsv4_read_device_flags() == 0
    res = O.decode_step(st, seqs=seqs, topk_override=st.given_topk if given else None)
    return CMP.check_step(st, res, gpu_results(ds), where=name), st, ds


@pytest.mark.parametrize("name", sorted(I.SMALL_CONFIGS))
def test_small_step_parity(lib, name):
    rep, _, _ = run_and_compare(name)
    assert rep["tokens"] == I.SMALL_CONFIGS[name].T


@pytest.mark.parametrize("name", ["small_c4_bf16", "small_c4_fp8", "small_c4_h128", "small_c4_f32"])
def test_small_attention_on_given_selection(lib, name):
    run_and_compare(name, given=True)


@pytest.mark.parametrize("name", ["tiny_c4_f32"])
def test_tiny_config_full_parity(lib, name):
    run_and_compare(name)


@pytest.mark.parametrize("name,seqs", [("csa_c4_bf16", [0, 17, 31]), ("hca_c128_bf16", [0, 21, 63]),
                                       ("csa_c4_fp8", [0, 77, 127]), ("csa_c4_1m", [0, 3]),
                                       ("csa_c4_mxfp4", [0, 13, 31]), ("csa_c4_cand", [0, 4, 5, 31]),
                                       ("csa_c4_src", [0, 9, 31])])
def test_full_size_sampled_parity(lib, name, seqs):
    rep, st, ds = run_and_compare(name, seqs=seqs)
    assert rep["tokens"] == len(seqs) * st.cfg.q_per_seq


def test_full_size_emitting_fold_parity(lib):
    """c128 with every sequence emitting a compressed entry this step (contexts multiple of 128)."""
    import dataclasses
    cfg = dataclasses.replace(I.CONFIGS["hca_c128_bf16"], name="hca_all_emit", B=8,
                              explicit_lens=tuple(65536 + 128 * k for k in range(8)))
    I.ALL_CONFIGS[cfg.name] = cfg
    try:
        run_and_compare(cfg.name, seqs=[0, 5])
    finally:
        del I.ALL_CONFIGS[cfg.name]


def test_bad_block_table_is_flagged_not_faulting(lib):
    """A block-table page outside the cache is skipped by the kernels and reported by the flags."""
    from deepseek_v4_hybrid_gb300.step import DeviceStep
    import deepseek_v4_hybrid_gb300 as M
    st = I.make_step(I.SMALL_CONFIGS["small_c4_bf16"])
    ds = DeviceStep(st)
    ds.run()
    torch.cuda.synchronize()
    assert M.dsv4_read_device_flags() == 0
    bad = ds.main_bt.clone()
    bad[0, 0] = ds.main_cache.shape[0] + 5
    ds.at_params.main_block_table = bad.data_ptr()
    ds.attention()
    torch.cuda.synchronize()
    assert M.dsv4_read_device_flags() & 1
    assert M.dsv4_read_device_flags() == 0       # flags clear after reading
    assert torch.isfinite(ds.out.float()).all()


@pytest.mark.parametrize("mode", ["all_ties", "negative"])
def test_topk_ties_and_negative_scores(lib, mode):
    """Every score equal (zero head weights: the lowest indices must win) and all-negative scores."""
    from deepseek_v4_hybrid_gb300.step import DeviceStep
    import deepseek_v4_hybrid_gb300 as M
    st = I.make_step(I.SMALL_CONFIGS["small_c4_bf16"])
    if mode == "all_ties":
        st.w_idx = np.zeros_like(st.w_idx)
    else:
        st.w_idx = -np.abs(st.w_idx) - 0.01
    ds = DeviceStep(st)
    ds.run()
    torch.cuda.synchronize()
    assert M.dsv4_read_device_flags() == 0
    res = O.decode_step(st)
    CMP.check_step(st, res, gpu_results(ds), where=mode)
    if mode == "all_ties":
        got = to_host(ds.topk_idx)
        for t in range(st.cfg.T):
            nc = O.n_compressed(int(st.positions[t]), st.cfg.ratio)
            m = min(nc, st.cfg.topk)
            assert np.array_equal(got[t][:m], np.arange(m))


@pytest.mark.parametrize("name", ["small_c4_bf16", "small_c128_bf16", "small_c4_fp8"])
@pytest.mark.parametrize("order", ["indexer_first", "compress_first"])
def test_after_independent_gives_the_same_caches(lib, name, order):
    """insert and compress with after_independent (start at once, wait for the kernel before them only
    before exiting) write exactly what they write when they wait first: right after the indexer call
    (indexer -> insert -> compress), and the insert right after the compressor (compress -> insert ->
    indexer, the order of the decode step when the compressor writes the index keys)."""
    from deepseek_v4_hybrid_gb300.step import DeviceStep
    import deepseek_v4_hybrid_gb300 as M
    st = I.make_step(I.SMALL_CONFIGS[name])
    out = {}
    for late in (False, True):
        ds = DeviceStep(st)
        if order == "indexer_first":
            ds.indexer()
            ds.insert(after_independent=late)
            ds.compress(after_independent=late)
        else:
            ds.compress()
            ds.insert(after_independent=late)
            ds.indexer()
        ds.attention()
        torch.cuda.synchronize()
        assert M.dsv4_read_device_flags() == 0
        out[late] = {k: to_host(getattr(ds, k)) for k in ("swa_cache", "main_cache", "state", "idx_cache",
                                                          "topk_idx", "out")
                     if getattr(ds, k, None) is not None}
    for k, v in out[False].items():
        assert np.array_equal(v, out[True][k]), k


def test_fp8_block_exponents_on_both_scaling_paths(lib):
    """fp8_ds_mla caches whose UE8M0 block exponents span 126..142: the attention kernel scales the
    codes with one bf16x2 multiply by 2^(e - 7) up to e = 134 and with two (2^120, then 2^(e - 127))
    above, so both paths meet rows of the same tile; the result must still match the oracle."""
    from deepseek_v4_hybrid_gb300.step import DeviceStep
    import deepseek_v4_hybrid_gb300 as M
    st = I.make_step(I.SMALL_CONFIGS["small_c4_fp8"])
    rng = np.random.default_rng(0xE8)
    for cache in (st.swa_cache, st.main_cache):
        sc = cache[..., I.FP8_SCALE_OFF:I.FP8_SCALE_OFF + 8]
        cache[..., I.FP8_SCALE_OFF:I.FP8_SCALE_OFF + 8] = rng.integers(126, 143, size=sc.shape, dtype=np.uint8)
    ds = DeviceStep(st, topk_override=st.given_topk)
    ds.run()
    torch.cuda.synchronize()
    assert M.dsv4_read_device_flags() == 0
    res = O.decode_step(st, topk_override=st.given_topk)
    g = gpu_results(ds)
    lse = g.pop("lse")
    CMP.check_step(st, res, g, where="fp8 exponents 126..142")
    # the logits reach about 1e5 here, and fp32 scores (576-term dot products) carry an absolute
    # error proportional to their size: the log-sum-exp is held to 2^-14 of its magnitude on top of
    # the usual 2e-3
    for t in res["tokens"]:
        ref = np.asarray(res["lse"][t], np.float64)
        assert np.all(np.abs(lse[t] - ref) <= 2e-3 + 2.0 ** -14 * np.abs(ref)), f"lse of token {t}"


@pytest.mark.parametrize("name", ["small_c4_bf16", "small_c4_fp8", "small_c4_f32"])
def test_kv_insert_with_rope(lib, name):
    """dsv4_kv_insert with a rotary table: each new row's dims 512..575 turned at its position, then
    encoded into the SWA cache (oracle kv_insert with positions and cos_sin)."""
    import deepseek_v4_hybrid_gb300 as M
    from deepseek_v4_hybrid_gb300.step import to_device
    st = I.make_step(I.SMALL_CONFIGS[name])
    cfg = st.cfg
    cache = to_device(st.swa_cache, "cuda")
    M.dsv4_kv_insert(to_device(st.kv_new, "cuda"), cfg.act_dtype, to_device(st.slot_mapping.astype(np.int64), "cuda"),
                     cache, cfg.cache_dtype, 64, positions=to_device(st.positions.astype(np.int32), "cuda"),
                     cos_sin=to_device(st.cos_sin, "cuda"))
    torch.cuda.synchronize()
    assert M.dsv4_read_device_flags() == 0
    swa = O.Paged(st.swa_cache)
    O.kv_insert(swa, st.kv_new, cfg.act_dtype, st.slot_mapping, cfg.cache_dtype, st.positions, st.cos_sin)
    got = to_host(cache)
    assert len(swa.written) == cfg.T
    for (page, off), row in swa.written.items():
        ok, _ = CMP.entry_error_ok(got[page, off], O.decode_rows(row, cfg.cache_dtype), cfg.cache_dtype)
        assert ok, (page, off)


def test_qprep_in_place_and_without_switches(lib):
    """The fused call with q_out = q (same head count) gives what it gives into a separate buffer, and
    with every switch off it copies the heads and zero-pads."""
    import deepseek_v4_hybrid_gb300 as M
    from deepseek_v4_hybrid_gb300.step import to_device
    st = I.make_step(I.SMALL_CONFIGS["small_c4_bf16"])
    cfg = st.cfg
    dev = lambda a: to_device(a, "cuda")  # noqa: E731
    q = dev(st.q)
    slots = dev(np.full(cfg.T, -1, np.int64))            # no kv stored
    cache = dev(st.swa_cache)
    sep = torch.empty_like(q)
    args = (cfg.act_dtype, dev(st.kv_new), slots, cache, cfg.cache_dtype, 64, dev(st.positions.astype(np.int32)),
            dev(st.cos_sin))
    M.dsv4_qnorm_rope_kv_insert(q, sep, *args, q_norm_weight=dev(st.q_norm_w))
    M.dsv4_qnorm_rope_kv_insert(q, q, *args, q_norm_weight=dev(st.q_norm_w))
    torch.cuda.synchronize()
    assert torch.equal(q.view(torch.int16), sep.view(torch.int16))
    padded = torch.empty((cfg.T, 96, 576), dtype=torch.bfloat16, device="cuda")
    q0 = dev(st.q)
    M.dsv4_qnorm_rope_kv_insert(q0, padded, *args, apply_q_norm=False, apply_q_rope=False, apply_kv_rope=False)
    torch.cuda.synchronize()
    assert M.dsv4_read_device_flags() == 0
    assert torch.equal(padded[:, :cfg.H].view(torch.int16), q0.view(torch.int16))
    assert torch.count_nonzero(padded[:, cfg.H:].float()) == 0


@pytest.mark.parametrize("name", ["small_c4_bf16", "small_c4_h128", "small_c4_fp8"])
def test_indexer_workspace_left_clean(lib, name):
    """Calls with workspace_zeroed = 1 (no memset) rely on every completed call clearing the histograms
    and counters it used: three calls in a row on one zero-filled workspace give the oracle's top-k
    sets each time as a call that clears the workspace first (whose parity the step tests check)."""
    import deepseek_v4_hybrid_gb300 as M
    from deepseek_v4_hybrid_gb300.step import DeviceStep
    st = I.make_step(I.SMALL_CONFIGS[name])
    ds = DeviceStep(st)
    assert ds.ix_params.workspace_zeroed == 1
    ds.compress()  # the keys this step's indexer reads
    outs = []
    for zeroed in (1, 1, 1, 0):
        ds.ix_params.workspace_zeroed = zeroed
        ds.indexer()
        torch.cuda.synchronize()
        assert M.dsv4_read_device_flags() == 0
        outs.append(to_host(ds.topk_idx).copy())
    for got in outs:
        assert np.array_equal(got, outs[-1])


def test_two_level_chain_source_feeds_consumer(lib):
    """The candidate source publishes its tokens' best blocks on the device; a later layer (its own keys
    and queries, the same positions) consumes exactly those lists: the consumer's selection matches the
    oracle given the same lists, and every selected entry lies in a published block."""
    import dataclasses
    from deepseek_v4_hybrid_gb300.step import DeviceStep
    src_cfg = I.SMALL_CONFIGS["small_c4_cand_src"]
    st_a = I.make_step(src_cfg)
    ds_a = DeviceStep(st_a)
    ds_a.run()
    torch.cuda.synchronize()
    assert lib.dsv4_read_device_flags() == 0
    published = to_host(ds_a.cand_blocks).copy()
    res_a = O.decode_step(st_a)
    for t in res_a["tokens"]:
        assert CMP.cand_blocks_match(published[t], res_a["scores"][t], src_cfg.cand_block, src_cfg.cand_topk)
    cons_cfg = dataclasses.replace(src_cfg, name="chain_consumer", cand_write=False, seed=src_cfg.seed + 99)
    st_b = I.make_step(cons_cfg)
    st_b.cand_in = published
    ds_b = DeviceStep(st_b)
    ds_b.run()
    torch.cuda.synchronize()
    assert lib.dsv4_read_device_flags() == 0
    res_b = O.decode_step(st_b)
    CMP.check_step(st_b, res_b, gpu_results(ds_b), where="chain consumer")
    sel = to_host(ds_b.topk_idx)
    for t in res_b["tokens"]:
        nc = len(res_b["scores"][t])
        if nc > cons_cfg.topk:
            blocks = set(published[t][published[t] >= 0].tolist())
            assert all(j // cons_cfg.cand_block in blocks for j in sel[t][sel[t] >= 0])
