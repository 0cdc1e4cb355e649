"""GPU decode path (Algorithm 2) against the CPU oracle, through the C ABI.

Both sides consume the same seeded compressed state (synth.make_state): the
library through shadowkv_load_state, the oracle directly.  Every step checks
  a7  the landmark logits P = q L^T / sqrt(d),
  a8  the selected chunks (tie-aware index rule),
  a9  the cache hit counts (exact) and, through the output, the fetched values,
  a10 the rebuilt keys RoPE(Gather(A, I) B),
  a11 the attention output (per-head relative error bound),
with the oracle's output computed on the GPU's selection once that selection
has been shown to be a valid top-k of the oracle's scores.
"""
import numpy as np
import pytest
import torch

from helpers import TOL, check_selection, head_errors, np64, oracle_state
from oracle import shadowkv_oracle as O
from sparse_rank_kv_gb300 import binding, build, synth
from sparse_rank_kv_gb300.synth import CONFIGS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    binding.lib()


SMALL = CONFIGS["llama_b1_s32k"].with_(
    name="small", b=2, h_q=8, h_kv=2, d=128, s=8000 + 64, c=8, r=64, k=37, o=6, w=64,
    theta=5e5, dtype="bf16", steps=6, seed=11)


def run_parity(cfg, steps=None, group="max", cache=True, bsel=None, rows=True, append=True,
               v_on_host=False, split=None, st=None, sels=None, opts=None):
    """Decode `steps` steps of `cfg` (state `st`, else a random one) and check
    each against the oracle; the selections are appended to `sels` if given;
    `opts` maps context options to values."""
    if st is None:
        st = synth.make_state(cfg, device="cuda")
    if v_on_host:
        st["v"] = st["v"].cpu()
    p = binding.make_params(cfg, group_reduce=binding.GROUP_MAX if group == "max" else binding.GROUP_SUM)
    ctx = binding.load_state(p, st)
    if not cache:
        ctx.set_option(binding.OPT_CACHE, 0)
    if split:
        ctx.set_option(binding.OPT_SPLIT_TOKENS, split)
    for o, v in (opts or {}).items():
        ctx.set_option(o, v)
    sl = slice(None) if bsel is None else slice(bsel, bsel + 1)
    dec = O.OracleDecoder(oracle_state(st, cfg, bsel), h_q=cfg.h_q, k=cfg.k, group_reduce=group,
                          key_dtype=cfg.dtype)
    b, h, hq, d, k, c, n = cfg.b, cfg.h_kv, cfg.h_q, cfg.d, cfg.k, cfg.c, cfg.n
    dt = synth.torch_dtype(cfg.dtype)
    T = cfg.steps if steps is None else steps
    outs, worst = [], 0.0
    for t in range(T):
        q = st["q"][t].contiguous()
        kn = st["k_new"][t].contiguous() if append else None
        vn = st["v_new"][t].contiguous() if append else None
        out = torch.empty(b, hq, d, dtype=dt, device="cuda")
        ctx.decode_step(q, kn, vn, out)
        torch.cuda.synchronize()
        sel = ctx.export("SEL").view(b, h, k).numpy()[sl]
        qn = np64(q[sl])
        P, S2, _ = dec.scores(qn)
        check_selection(sel, S2, k, what=f"step {t} selection")
        if sels is not None:
            sels.append(sel.copy())
        res = dec.step(qn, np64(kn[sl]) if append else None, np64(vn[sl]) if append else None,
                       force_sel=sel)
        err = head_errors(np64(out[sl]), res.out)
        worst = max(worst, float(err.max()))
        assert err.max() <= TOL[cfg.dtype], f"step {t}: output error {err.max():.3g}"
        hits = ctx.export("HITS").view(b, h).numpy()[sl]
        want = res.hits if cache else np.zeros_like(res.hits)   # cache off: all refetched
        assert np.array_equal(hits, want), f"step {t}: hits {hits} vs {want}"
        if rows:
            lg = ctx.export("LOGITS").view(b, hq, n).numpy()[sl].astype(np.float64)
            m = ~np.isnan(res.P)
            scale = np.abs(res.P[m]).max()
            assert np.abs(lg[m] - res.P[m]).max() <= 1e-5 * scale + 1e-6, f"step {t}: logits"
            ks = np64(ctx.export("K_SPARSE").view(b, h, k * c, d)[sl])
            kref = res.K_sparse
            tol = (1e-5 if cfg.dtype == "f32" else 8e-3) * np.abs(kref).max()
            assert np.abs(ks - kref).max() <= tol, f"step {t}: rebuilt keys"
        outs.append(out.clone())
    ctx.check()
    stats = ctx.stats()
    return outs, ctx, stats, worst


@pytest.mark.parametrize("cfg", [
    SMALL.with_(seed=42),
    SMALL.with_(r=48, seed=43),                       # last K block half out of range
    SMALL.with_(c=16, k=20, seed=44),                 # 16-row chunk boxes
    SMALL.with_(d=64, theta=1e4, seed=45),            # N = 64
    SMALL.with_(h_q=16, seed=48),                     # G = 8 (x8 TMEM loads)
    SMALL.with_(h_q=2, seed=49),                      # G = 1
], ids=["r64", "r48", "c16", "d64", "g8", "g1"])
def test_tensor_core_kernels_match_cuda_core_kernels(cfg):
    """The tcgen05 kernels and the fp32 CUDA-core kernels compute the same
    landmark logits (fp32 sums of exact bf16 products) and the same
    RoPE(Gather(A, I) B) (both round an fp32 result to bf16)."""
    st = synth.make_state(cfg, device="cuda")
    got = []
    for simt in (0, 1):
        ctx = binding.load_state(binding.make_params(cfg), st)
        ctx.set_option(binding.OPT_CUDA_CORES, simt)
        out = torch.empty(cfg.b, cfg.h_q, cfg.d, dtype=torch.bfloat16, device="cuda")
        ctx.decode_step(st["q"][0], st["k_new"][0], st["v_new"][0], out)
        torch.cuda.synchronize()
        ctx.check()
        got.append((ctx.export("K_SPARSE").float(), out.float().cpu(), ctx.export("LOGITS")))
    (k_tc, o_tc, l_tc), (k_simt, o_simt, l_simt) = got
    assert (l_tc - l_simt).abs().max() <= 1e-5 * l_simt.abs().max()
    assert (k_tc - k_simt).abs().max() <= 2.0 ** -7 * k_simt.abs().max()
    assert (o_tc - o_simt).abs().max() <= 1e-2 * o_simt.abs().max()


def test_tiny_fp32_all_steps():
    _, _, stats, worst = run_parity(CONFIGS["tiny_f32_s1k"])
    assert stats.steps == 4 and worst <= TOL["f32"]


def test_small_bf16_ragged_tiles():
    # n = 1000 (not a multiple of the 128-landmark score tile), k*c = 296 rows
    # (not a multiple of the 64-row rebuild tile), ragged attention splits
    run_parity(SMALL)


@pytest.mark.parametrize("G", [1, 2, 8])
def test_group_sizes(G):
    run_parity(SMALL.with_(h_q=2 * G, seed=20 + G), steps=3)


def test_head_dim_64_bf16():
    run_parity(SMALL.with_(d=64, theta=1e4, seed=31), steps=3)


def test_group_reduce_sum_reading():
    run_parity(SMALL.with_(seed=32), steps=3, group="sum")


def test_no_local_prompt_window_and_no_outliers():
    run_parity(SMALL.with_(s=8000, w=0, o=0, seed=33), steps=3)


def test_decode_without_appending():
    run_parity(SMALL.with_(seed=34), steps=3, append=False)


def test_k_one_and_k_all_candidates():
    run_parity(SMALL.with_(k=1, seed=35), steps=3)
    cfg = SMALL.with_(s=600 * 8 + 64, o=4, seed=36)
    run_parity(cfg.with_(k=cfg.n - cfg.o), steps=3)


def test_split_size_variants():
    run_parity(SMALL.with_(seed=37), steps=2, split=32)
    run_parity(SMALL.with_(seed=37), steps=2, split=256)


def test_values_from_host_memory():
    run_parity(SMALL.with_(seed=38), steps=3, v_on_host=True)


@pytest.mark.parametrize("in_attn", [0, 1], ids=["rebuild_launch", "rebuild_in_attention"])
def test_cache_is_lossless(in_attn):
    """The set-difference cache changes only what crosses the host link.  With
    the cache on and forced off every step attends bit-identical data: the
    same chunks, the same rebuilt keys and the same values for them.  The
    outputs agree to the rounding of the attention's sums: cache hits and
    misses are summed in different partials (hits first), so the fp32 sums
    may round differently before the bf16 output (at most 2 bf16 ulps of a
    head's largest value)."""
    cfg = SMALL.with_(steps=8, seed=39)
    st = synth.make_state(cfg, device="cuda")
    b, h, hq, d, k, c = cfg.b, cfg.h_kv, cfg.h_q, cfg.d, cfg.k, cfg.c
    ctxs = [binding.load_state(binding.make_params(cfg), st) for _ in range(2)]
    ctxs[1].set_option(binding.OPT_CACHE, 0)
    for ctx in ctxs:
        ctx.set_option(binding.OPT_REBUILD_IN_ATTENTION, in_attn)
        assert ctx.layout()["rebuild_in_attention"] == in_attn
    dt = synth.torch_dtype(cfg.dtype)

    def attended(ctx):
        sel = ctx.export("SEL").view(b, h, k)
        slots = ctx.export("SEL_SLOT").view(b, h, k).long()
        kspa = ctx.export("K_SPARSE").view(b, h, k * c, d)
        vslot = ctx.export("SLOT_V").view(b, h, k, c, d)
        vsel = torch.gather(vslot, 2, slots[..., None, None].expand(b, h, k, c, d))
        return sel, kspa, vsel

    for t in range(cfg.steps):
        outs = []
        for ctx in ctxs:
            out = torch.empty(b, hq, d, dtype=dt, device="cuda")
            ctx.decode_step(st["q"][t].contiguous(), st["k_new"][t].contiguous(),
                            st["v_new"][t].contiguous(), out)
            torch.cuda.synchronize()
            outs.append(out)
        (s0, k0, v0), (s1, k1, v1) = attended(ctxs[0]), attended(ctxs[1])
        assert torch.equal(s0, s1), f"step {t}: selections differ"
        assert torch.equal(k0, k1), f"step {t}: rebuilt keys differ"
        assert torch.equal(v0, v1), f"step {t}: values of the selected chunks differ"
        err = head_errors(np64(outs[0]), np64(outs[1]))
        assert err.max() <= 8e-3, f"step {t}: outputs differ by {err.max():.3g}"
    for ctx in ctxs:
        ctx.check()
    st_on, st_off = ctxs[0].stats(), ctxs[1].stats()
    assert st_off.hits == 0 and st_off.misses == cfg.steps * cfg.b * cfg.h_kv * cfg.k
    assert st_on.hits > 0 and st_on.hits + st_on.misses == st_off.misses


def test_full_size_32k():
    run_parity(CONFIGS["llama_b1_s32k"])


@pytest.mark.parametrize("name,bsel,steps", [
    ("llama_b8_s128k", 5, 6),
    ("llama_b48_s60k", 37, 4),
    ("llama_b2_s256k", 1, 5),
])
def test_full_size_sampled_sequence(name, bsel, steps):
    """The full-size workloads in the benchmark's launch configuration; the
    oracle recomputes one sequence of the batch."""
    run_parity(CONFIGS[name], steps=steps, bsel=bsel, rows=False)


@pytest.mark.parametrize("cfg", [
    SMALL.with_(seed=50),
    SMALL.with_(r=48, seed=51),                       # last K block half out of range
    SMALL.with_(c=16, k=20, seed=52),                 # 16-row chunks: 8 per item
    SMALL.with_(b=6, h_kv=8, h_q=32, k=64, seed=53),  # 48 heads: more tiles than rebuild CTAs
], ids=["r64", "r48", "c16", "h48"])
def test_rebuild_inside_the_attention_launch(cfg):
    """SKV_OPT_REBUILD_IN_ATTENTION: the first CTAs of the attention's launch
    rebuild the missed chunks' keys into their cache slots, then take
    attention items; each missed chunk's item waits for its own keys and
    values.  Selections, hits, rebuilt keys and outputs against the oracle on
    every step."""
    _, ctx, _, _ = run_parity(cfg, opts={binding.OPT_REBUILD_IN_ATTENTION: 1})
    assert ctx.layout()["rebuild_in_attention"] == 1


def test_rebuild_inside_the_attention_launch_full_size():
    """The same at batch 8, 128K (the oracle recomputes one sequence)."""
    _, ctx, _, _ = run_parity(CONFIGS["llama_b8_s128k"], steps=4, bsel=2, rows=False,
                              opts={binding.OPT_REBUILD_IN_ATTENTION: 1})
    assert ctx.layout()["rebuild_in_attention"] == 1


@pytest.mark.parametrize("q_sigma", [2.0, 0.02], ids=["large_moves", "small_moves"])
def test_selection_threshold_carried_between_steps(q_sigma):
    """The selection's first threshold try is the previous step's k-th
    largest S2 minus a margin; a try that leaves fewer than k chunks at or
    above it falls back to the threshold from the bounds.  With large query
    moves most tries fail, with small ones most succeed: every selection is
    checked against the oracle either way."""
    run_parity(SMALL.with_(q_sigma=q_sigma, steps=6, seed=60))


def test_selections_repeat_after_a_rewind():
    """A rewind empties the cache and drops the carried threshold: the same
    steps again give the same selections (the carried threshold changes how
    the top k is found, never which chunks it holds)."""
    cfg = SMALL.with_(steps=5, seed=61)
    st = synth.make_state(cfg, device="cuda")
    ctx = binding.load_state(binding.make_params(cfg), st)
    dt = synth.torch_dtype(cfg.dtype)
    runs = []
    for _ in range(2):
        sels = []
        for t in range(cfg.steps):
            out = torch.empty(cfg.b, cfg.h_q, cfg.d, dtype=dt, device="cuda")
            ctx.decode_step(st["q"][t].contiguous(), st["k_new"][t].contiguous(), st["v_new"][t].contiguous(), out)
            torch.cuda.synchronize()
            sels.append(ctx.export("SEL").clone())
        runs.append(sels)
        ctx.rewind()
    ctx.check()
    for t in range(cfg.steps):
        assert torch.equal(runs[0][t], runs[1][t]), f"step {t}: selections differ after the rewind"


def test_max_new_is_enforced():
    cfg = SMALL.with_(steps=2, seed=40)
    st = synth.make_state(cfg, device="cuda")
    ctx = binding.load_state(binding.make_params(cfg), st)
    out = torch.empty(cfg.b, cfg.h_q, cfg.d, dtype=torch.bfloat16, device="cuda")
    for t in range(2):
        ctx.decode_step(st["q"][t], st["k_new"][t], st["v_new"][t], out)
    with pytest.raises(binding.ShadowKVError) as ei:
        ctx.decode_step(st["q"][0], st["k_new"][0], st["v_new"][0], out)
    assert ei.value.code == 6
    ctx.decode_step(st["q"][0], None, None, out)   # no append: still fine
    ctx.check()


def test_bad_outlier_ids_are_reported():
    cfg = SMALL.with_(seed=41)
    st = synth.make_state(cfg, device="cuda")
    st["outlier_ids"][0, 0, 1] = st["outlier_ids"][0, 0, 0]   # duplicate
    with pytest.raises(binding.ShadowKVError) as ei:
        binding.load_state(binding.make_params(cfg), st)
    assert ei.value.code == 4


@pytest.mark.parametrize("cfg", [SMALL.with_(r=48, seed=46), SMALL.with_(c=16, k=20, seed=47)],
                         ids=["r48", "c16"])
def test_rebuild_shape_variants_against_oracle(cfg):
    run_parity(cfg, steps=3)


def test_selection_with_massive_ties():
    """Most landmarks equal: the sampled threshold admits far more than 2048
    survivors, so the radix select decides; ties go to the lower index."""
    cfg = CONFIGS["llama_b1_s32k"].with_(b=1, steps=3, seed=60)
    st = synth.make_state(cfg, device="cuda")
    hot = st["L"][:, :, :20].clone()
    st["L"].zero_()
    st["L"][:, :, 100:120] = hot
    run_parity(cfg, steps=3, st=st)


def test_selection_ties_at_the_threshold():
    """Landmarks in identical triples at 128K (sampled threshold): the k-th
    key has equal keys on both sides of the cut, and the selection takes the
    lowest-index copies of a triple first."""
    cfg = CONFIGS["llama_b8_s128k"].with_(b=1, steps=3, seed=61)
    st = synth.make_state(cfg, device="cuda")
    m = (cfg.n - cfg.o) // 3 * 3
    L = st["L"]
    L[:, :, 1:m:3] = L[:, :, 0:m:3]
    L[:, :, 2:m:3] = L[:, :, 0:m:3]
    # the outliers lie past the triples, so every copy of a triple is a candidate
    st["outlier_ids"][:] = torch.arange(m, m + cfg.o, device="cuda", dtype=torch.int32)
    sels = []
    run_parity(cfg, steps=3, rows=False, st=st, sels=sels)
    for t, sel in enumerate(sels):
        for row in sel.reshape(-1, cfg.k):
            chosen = set(row.tolist())
            for j in row:
                if j < m:
                    t0 = j - j % 3
                    assert all(x in chosen for x in range(t0, j)), f"step {t}: chunk {j} without its lower copies"


def test_steps_do_not_run_into_wait_limits():
    """Every bounded wait in the kernels gives up after 2 s: a step that takes
    that long has a wait that never completes, even when nothing is flagged."""
    import time
    cfg = CONFIGS["llama_b8_s128k"].with_(b=2, steps=6, seed=62)
    st = synth.make_state(cfg, device="cuda")
    ctx = binding.load_state(binding.make_params(cfg), st)
    out = torch.empty(cfg.b, cfg.h_q, cfg.d, dtype=torch.bfloat16, device="cuda")
    for t in range(cfg.steps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ctx.decode_step(st["q"][t], st["k_new"][t], st["v_new"][t], out)
        torch.cuda.synchronize()
        assert time.perf_counter() - t0 < 0.5, f"step {t} took {time.perf_counter() - t0:.2f} s"
    ctx.check()


def test_misaligned_queries_are_rejected_before_any_work():
    """q is read in place through tensor maps: a q that is not 16-byte aligned
    is refused with an argument error and the context's state is untouched."""
    cfg = SMALL.with_(steps=2, seed=63)
    st = synth.make_state(cfg, device="cuda")
    ctx = binding.load_state(binding.make_params(cfg), st)
    out = torch.empty(cfg.b, cfg.h_q, cfg.d, dtype=torch.bfloat16, device="cuda")
    q = st["q"][0].contiguous()
    buf = torch.empty(q.numel() + 8, dtype=q.dtype, device="cuda")
    qm = buf[1:1 + q.numel()].view_as(q)
    qm.copy_(q)
    before = ctx.stats()
    with pytest.raises(binding.ShadowKVError) as ei:
        ctx.decode_step(qm, st["k_new"][0], st["v_new"][0], out)
    assert ei.value.code == 1
    after = ctx.stats()
    assert after.hits == before.hits and after.misses == before.misses and after.launches == before.launches
    ctx.decode_step(q, st["k_new"][0], st["v_new"][0], out)
    ctx.check()


@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_buffer_step_equals_device_step(pinned):
    """shadowkv_decode_step_host (inputs and output in host memory) runs the
    same step as shadowkv_decode_step on device buffers: identical selections
    and hits, bit-identical outputs, over steps with a warm cache."""
    cfg = SMALL.with_(steps=5, seed=64)
    st = synth.make_state(cfg, device="cuda")
    p = binding.make_params(cfg)
    dev_ctx, host_ctx = binding.load_state(p, st), binding.load_state(p, st)
    dt = synth.torch_dtype(cfg.dtype)
    host = lambda t: t.cpu().pin_memory() if pinned else t.cpu()
    out_h = host(torch.empty(cfg.b, cfg.h_q, cfg.d, dtype=dt))
    stream = torch.cuda.current_stream()
    for t in range(cfg.steps):
        out_d = torch.empty(cfg.b, cfg.h_q, cfg.d, dtype=dt, device="cuda")
        dev_ctx.decode_step(st["q"][t], st["k_new"][t], st["v_new"][t], out_d)
        host_ctx.decode_step_host(host(st["q"][t]), host(st["k_new"][t]), host(st["v_new"][t]), out_h, stream)
        torch.cuda.synchronize()
        for f in ("SEL", "HITS"):
            assert torch.equal(dev_ctx.export(f), host_ctx.export(f)), f"step {t}: {f}"
        assert torch.equal(out_d.cpu(), out_h), f"step {t}: outputs differ"
    dev_ctx.check()
    host_ctx.check()
