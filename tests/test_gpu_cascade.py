"""Cascade decode (shared prompt prefixes computed once per group) against the oracle.

The cascade splits each member's attention into its group's shared pages (prefix kernel,
once for all members) and its own pages (decode kernel), merged by the combine kernel; the
result must be the attention over all of the request's tokens, as the oracle computes it from
the request's contiguous tokens."""
import numpy as np
import pytest
import torch

import paged_kv_cache_271_gb300 as pkv
import workloads
from gpu_harness import GroupScenario, oracle_groups_expected

pytestmark = pytest.mark.gpu

TOL = 1e-2  # bf16 inputs and P rounded to bf16 in both tensor-core products


def _cascade(sc, groups, step=False, out=None, workspace=None):
    w = sc.w
    if step:
        return pkv.cascade_decode_step(sc.q, sc.k_new, sc.v_new, sc.cache.k, sc.cache.v,
                                       sc.block_tables, sc.context_lens, w.scale, groups,
                                       out=out, workspace=workspace)
    return pkv.cascade_decode_attention(sc.q, sc.cache.k, sc.cache.v, sc.block_tables,
                                        sc.context_lens, w.scale, groups, out=out,
                                        workspace=workspace)


def _check_no_error():
    assert pkv.device_error() == 0


def _case(G, h_kv=2, seed=11, groups=((5, 7, 1, 40), (2, 3, 1, 20)), singles=((1, 60),) * 3):
    return workloads.prefix_groups("cascade_g%d" % G, workloads.BASE_SEED + 500 + seed, G * h_kv,
                                   h_kv, 128, list(groups), list(singles))


@pytest.fixture(autouse=True, params=[1, 2], ids=["fold_in_decode", "fold_in_combine"])
def overlap_mode(request):
    # the own-page decode alongside the prefix kernel, folding the prefix partials itself (1)
    # or leaving them to the combine kernel (2)
    pkv.cascade_set_overlap(request.param)
    yield request.param
    pkv.cascade_set_overlap(2)


@pytest.fixture(params=[1, 2], ids=["prefix_mma_sync", "prefix_tcgen05"])
def prefix_kernel(request):
    pkv.cascade_set_prefix_kernel(request.param)
    yield request.param
    pkv.cascade_set_prefix_kernel(0)


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("kernel", [1, 2])
def test_cascade_matches_oracle(G, kernel, prefix_kernel):
    w = _case(G)
    sc = GroupScenario(w)
    sc.append()
    groups = pkv.cascade_groups(sc.bt_host, sc.cl_host).to(sc.q.device)
    assert groups.n_groups == 2 and sorted(groups.prefix_pages.tolist()) == [2, 5]
    pkv.device_error()
    pkv.decode_set_kernel(kernel)
    try:
        out = _cascade(sc, groups)
    finally:
        pkv.decode_set_kernel(0)
    torch.cuda.synchronize()
    _check_no_error()
    ref = oracle_groups_expected(w)
    err = np.abs(out.float().cpu().numpy() - ref).max()
    assert err < TOL, err


def test_cascade_step_equals_append_then_cascade_and_oracle(prefix_kernel):
    w = _case(4, h_kv=4, seed=12)
    sc = GroupScenario(w)
    groups = pkv.cascade_groups(sc.bt_host, sc.cl_host).to(sc.q.device)
    k0, v0 = sc.cache.k.clone(), sc.cache.v.clone()
    pkv.device_error()
    fused = _cascade(sc, groups, step=True).clone()
    k1, v1 = sc.cache.k.clone(), sc.cache.v.clone()
    sc.cache.k.copy_(k0)
    sc.cache.v.copy_(v0)
    sc.append()
    split = _cascade(sc, groups)
    torch.cuda.synchronize()
    _check_no_error()
    assert torch.equal(sc.cache.k.view(torch.uint8), k1.view(torch.uint8))
    assert torch.equal(sc.cache.v.view(torch.uint8), v1.view(torch.uint8))
    assert torch.equal(fused, split)
    err = np.abs(fused.float().cpu().numpy() - oracle_groups_expected(w)).max()
    assert err < TOL, err


@pytest.mark.parametrize("chunk", [1, 3, 8, 32, 70])
def test_cascade_prefix_chunking_and_ragged_row_tiles(chunk, prefix_kernel):
    # 70 shared pages split into several chunks (or one of 18 tiles: the copy ring and the
    # page masks wrap several times); 17 members x 4 heads = 68 rows: a ragged second row
    # tile; singles long enough to need the split decode too
    w = _case(4, h_kv=2, seed=13, groups=((70, 17, 1, 90),), singles=((700, 1400),) * 2)
    sc = GroupScenario(w)
    sc.append()
    groups = pkv.cascade_groups(sc.bt_host, sc.cl_host).to(sc.q.device)
    pkv.cascade_set_prefix_chunk_pages(chunk)
    pkv.device_error()
    try:
        assert pkv.cascade_prefix_chunk_pages(2, 8, groups) == chunk
        out = _cascade(sc, groups)
        torch.cuda.synchronize()
    finally:
        pkv.cascade_set_prefix_chunk_pages(0)
    _check_no_error()
    err = np.abs(out.float().cpu().numpy() - oracle_groups_expected(w)).max()
    assert err < TOL, err


@pytest.mark.parametrize("own_pages", [(1, 90), (300, 700)], ids=["one_own_chunk", "own_chunks"])
def test_cascade_overlap_on_and_off_agree(own_pages, prefix_kernel):
    # the own-page decode as a dependent launch of the prefix kernel (waiting for it only
    # before the fold) and after it: the same kernels, so the same bits
    lo, hi = own_pages
    w = _case(4, h_kv=4, seed=14, groups=((40, 9, lo, hi), (3, 5, lo, hi)),
              singles=((lo, hi),) * 3)
    sc = GroupScenario(w)
    sc.append()
    groups = pkv.cascade_groups(sc.bt_host, sc.cl_host).to(sc.q.device)
    pkv.device_error()
    outs = []
    try:
        for mode in (0, 1, 2):
            pkv.cascade_set_overlap(mode)
            outs.append(_cascade(sc, groups).clone())
            torch.cuda.synchronize()
            _check_no_error()
    finally:
        pkv.cascade_set_overlap(2)
    assert torch.equal(outs[0], outs[1])  # the same kernels in the same order
    ref = oracle_groups_expected(w)
    for o in outs[1:]:  # (mode 2 merges the same partials in another order)
        err = np.abs(o.float().cpu().numpy() - ref).max()
        assert err < TOL, err


def test_cascade_host_step_equals_device_step():
    # the step from host memory (queries, new rows, tables and lengths packed in one pinned
    # buffer, the groups found on the host): same output and pool bytes as the device step
    w = _case(4, h_kv=4, seed=15)
    a = GroupScenario(w)
    groups = pkv.cascade_groups(a.bt_host, a.cl_host).to(a.q.device)
    pkv.device_error()
    out_a = _cascade(a, groups, step=True).clone()
    b = GroupScenario(w)
    hs = pkv.HostStep(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, b.block_tables.shape[1])
    hs.q_host.copy_(b.q.cpu())
    hs.k_new_host.copy_(b.k_new.cpu())
    hs.v_new_host.copy_(b.v_new.cpu())
    hs.block_tables_host.copy_(b.block_tables.cpu())
    hs.context_lens_host.copy_(b.context_lens.cpu())
    g_host = pkv.cascade_groups(hs.block_tables_host.numpy(), hs.context_lens_host.numpy())
    ws = torch.zeros(pkv.cascade_workspace_size(w.batch, w.num_q_heads, w.num_kv_heads,
                                                w.head_dim, b.block_tables.shape[1], g_host),
                     dtype=torch.uint8, device=b.q.device)
    out_b = hs.step(b.cache.k, b.cache.v, w.scale, workspace=ws, groups=g_host.to(b.q.device))
    torch.cuda.synchronize()
    _check_no_error()
    assert torch.equal(out_a.cpu(), out_b)
    assert torch.equal(a.cache.k.view(torch.uint8), b.cache.k.view(torch.uint8))
    assert torch.equal(a.cache.v.view(torch.uint8), b.cache.v.view(torch.uint8))
    err = np.abs(out_b.float().numpy() - oracle_groups_expected(w)).max()
    assert err < TOL, err


@pytest.mark.parametrize("grouped", [True, False], ids=["groups", "no_group"])
def test_packed_cascade_step_equals_device_step(grouped):
    # one library call from host memory: groups found on the host from the packed tables,
    # one copy in, the cascade step, one copy out
    w = _case(4, h_kv=4, seed=16, groups=((6, 9, 1, 60), (3, 4, 1, 30)) if grouped else (),
              singles=((1, 60),) * (3 if grouped else 7))
    a = GroupScenario(w)
    g_a = pkv.cascade_groups(a.bt_host, a.cl_host)
    assert (g_a.n_groups > 0) == grouped
    pkv.device_error()
    if grouped:
        out_a = _cascade(a, g_a.to(a.q.device), step=True).clone()
    else:
        out_a = pkv.paged_decode_step(a.q, a.k_new, a.v_new, a.cache.k, a.cache.v,
                                      a.block_tables, a.context_lens, w.scale).clone()
    b = GroupScenario(w)
    hs = pkv.HostStep(w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim,
                      b.block_tables.shape[1], cascade=True)
    hs.q_host.copy_(b.q.cpu())
    hs.k_new_host.copy_(b.k_new.cpu())
    hs.v_new_host.copy_(b.v_new.cpu())
    hs.block_tables_host.copy_(b.block_tables.cpu())
    hs.context_lens_host.copy_(b.context_lens.cpu())
    try:  # without a workspace: refused before anything runs, when the step needs one
        hs.cascade_step(b.cache.k, b.cache.v, w.scale, None)
        refused = False
    except pkv.PkvError:
        refused = True
    assert refused == (hs.workspace_needed > 0)
    ws = torch.zeros(max(hs.workspace_needed, 16), dtype=torch.uint8, device=b.q.device)
    out_b = hs.cascade_step(b.cache.k, b.cache.v, w.scale, ws)
    torch.cuda.synchronize()
    _check_no_error()
    assert hs.n_groups == g_a.n_groups
    assert torch.equal(out_a.cpu(), out_b)
    assert torch.equal(a.cache.k.view(torch.uint8), b.cache.k.view(torch.uint8))
    assert torch.equal(a.cache.v.view(torch.uint8), b.cache.v.view(torch.uint8))
    err = np.abs(out_b.float().numpy() - oracle_groups_expected(w)).max()
    assert err < TOL, err


def test_cascade_with_empty_suffix_and_no_groups(prefix_kernel):
    # a member whose context ends exactly at the end of the shared pages (attention only):
    # its own part is empty and the merge takes the prefix partials alone
    w = _case(4, h_kv=2, seed=14, groups=((3, 4, 1, 30),), singles=((1, 9),))
    sc = GroupScenario(w)
    sc.append()
    ref = oracle_groups_expected(w)
    groups = pkv.cascade_groups(sc.bt_host, sc.cl_host)
    # trim one member's context to the shared pages: still a valid cascade for attention
    b = int(groups.group_members[0])
    cl = sc.cl_host.copy()
    cl[b] = 16 * int(groups.prefix_pages[0])
    sc.context_lens.copy_(torch.from_numpy(cl))
    groups.to(sc.q.device)
    pkv.device_error()
    out = _cascade(sc, groups)
    plain = pkv.paged_decode_attention(sc.q, sc.cache.k, sc.cache.v, sc.block_tables,
                                       sc.context_lens, w.scale)
    torch.cuda.synchronize()
    _check_no_error()
    assert (out.float() - plain.float()).abs().max().item() < TOL
    others = [i for i in range(w.batch) if i != b]
    err = np.abs(out.float().cpu().numpy()[others] - ref[others]).max()
    assert err < TOL, err
    # no group at all: exactly the plain decode
    none = pkv.cascade_groups(sc.bt_host, sc.cl_host, min_members=w.batch + 1).to(sc.q.device)
    assert none.n_groups == 0
    assert torch.equal(_cascade(sc, none), plain)


def test_cascade_flags_members_that_do_not_cover_the_prefix(prefix_kernel):
    w = _case(4, h_kv=2, seed=15, groups=((3, 4, 5, 30),), singles=())
    sc = GroupScenario(w)
    sc.append()
    groups = pkv.cascade_groups(sc.bt_host, sc.cl_host)
    cl = sc.cl_host.copy()
    cl[int(groups.group_members[1])] = 20  # shorter than the 48 shared positions
    sc.context_lens.copy_(torch.from_numpy(cl))
    groups.to(sc.q.device)
    pkv.device_error()
    _cascade(sc, groups)
    assert pkv.device_error() & pkv.DEVERR_BAD_GROUP


def test_cascade_prefix_sharing_full_size_sampled(prefix_kernel):
    # 128 requests on one 2000-token prefix (125 pages), own suffixes U[5, 200]
    w = workloads.prefix_sharing()
    from gpu_harness import Scenario, oracle_expected
    sc = Scenario(w)
    sc.append()
    bt = sc.block_tables.cpu().numpy()
    groups = pkv.cascade_groups(bt, sc.context_lens.cpu().numpy()).to(sc.q.device)
    assert groups.n_groups == 1 and int(groups.prefix_pages[0]) == 125
    pkv.device_error()
    out = pkv.cascade_decode_attention(sc.q, sc.cache.k, sc.cache.v, sc.block_tables,
                                       sc.context_lens, w.scale, groups)
    plain = sc.decode()
    torch.cuda.synchronize()
    _check_no_error()
    assert (out.float() - plain.float()).abs().max().item() < TOL
    rng = np.random.default_rng(5)
    pairs = np.stack([rng.integers(0, w.batch, 48), rng.integers(0, w.num_q_heads, 48)], 1)
    ref = oracle_expected(w, pairs=pairs)
    got = out.float().cpu().numpy()[pairs[:, 0], pairs[:, 1]]
    assert np.abs(got - ref).max() < TOL


@pytest.mark.parametrize("own_chunk", [1, 2])
def test_cascade_members_with_several_own_chunks(own_chunk, prefix_kernel):
    # own pages split into chunks of 1-2 pages: every member's chunks write partials after its
    # prefix partials and the last chunk to finish merges them all (in place)
    w = _case(8, h_kv=2, seed=16, groups=((4, 5, 20, 70), (9, 3, 40, 90)), singles=((30, 200),))
    sc = GroupScenario(w)
    sc.append()
    groups = pkv.cascade_groups(sc.bt_host, sc.cl_host).to(sc.q.device)
    pkv.decode_set_chunk_pages(own_chunk)
    pkv.device_error()
    try:
        outs = [_cascade(sc, groups).clone() for _ in range(2)]  # counters reset between calls
        torch.cuda.synchronize()
    finally:
        pkv.decode_set_chunk_pages(0)
    _check_no_error()
    assert torch.equal(outs[0], outs[1])
    err = np.abs(outs[0].float().cpu().numpy() - oracle_groups_expected(w)).max()
    assert err < TOL, err


@pytest.mark.parametrize("chunk", [0, 3], ids=["default_chunks", "chunks_of_3"])
def test_cascade_without_page_ids_reads_the_first_members_row(chunk, prefix_kernel):
    # groups given without their shared page ids: the prefix kernel reads the ids from the
    # first member's table row instead; the same pages, so the same bits as with the ids
    w = _case(4, h_kv=2, seed=17, groups=((70, 17, 1, 90), (5, 3, 1, 40)),
              singles=((1, 60),) * 2)
    sc = GroupScenario(w)
    sc.append()
    g = pkv.cascade_groups(sc.bt_host, sc.cl_host)
    assert g.prefix_page_ids is not None
    with_ids = g.to(sc.q.device)
    bare = pkv.CascadeGroups(g.group_of, g.prefix_pages, g.group_offsets, g.group_members,
                             g.max_members, g.max_prefix_pages, g.max_own_pages,
                             g.own_start).to(sc.q.device)
    assert bare.prefix_page_ids is None and bare.desc().prefix_page_ids is None
    pkv.cascade_set_prefix_chunk_pages(chunk)
    pkv.device_error()
    try:
        a = _cascade(sc, with_ids).clone()
        b = _cascade(sc, bare).clone()
        torch.cuda.synchronize()
    finally:
        pkv.cascade_set_prefix_chunk_pages(0)
    _check_no_error()
    assert torch.equal(a, b)
    err = np.abs(b.float().cpu().numpy() - oracle_groups_expected(w)).max()
    assert err < TOL, err
