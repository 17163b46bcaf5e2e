"""GPU tests of the extended entry point: max_prob, packed documents (variable length),
the per-document dense fallback, and the checks on the offset tables."""
import math

import numpy as np
import pytest

import oracle
import synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import softmax_threshold_tile_gb300 as blasst
    blasst.build_library()
    blasst.load_library()
    yield
    torch.cuda.synchronize()


def _blasst():
    import softmax_threshold_tile_gb300 as blasst
    return blasst


def _clear_error():
    st, word = _blasst().blasst_device_error(clear=True)
    return word


@pytest.mark.parametrize("name,factor", [("tiny_1024", 0.0), ("tiny_1024", 2.0), ("dit_8192_g2", 16.0)])
def test_max_prob_matches_oracle(name, factor):
    import torch
    w = synth.WORKLOADS[name]
    q, k, v = synth.make_qkv(w)
    qd, kd, vd = (parity.to_device(x) for x in (q, k, v))
    res = _blasst().attn_fwd(qd, kd, vd, factor, want_mask=True, want_max_prob=True)
    torch.cuda.synchronize()
    assert _clear_error() == 0
    mask = res.skip_mask.cpu().numpy()
    mp = res.max_prob.cpu().numpy()
    units = parity.sample_units(w.B, w.H, w.S, heads=(0, w.H - 1), qtiles=(0, 1, w.S // 256, w.S // 128 - 1))
    m_in = np.stack([mask[b, h, t] for b, h, t in units])
    ref = oracle.skip_softmax_attn(q, k, v, 1 / math.sqrt(w.d), factor, units=units, mask_in=m_in, threads=parity.host_threads())
    for u, (b, h, t) in enumerate(units):
        got = mp[b, h, t * 128:(t + 1) * 128]
        np.testing.assert_allclose(got, ref["max_prob"][u], rtol=2e-3, atol=1e-6)
    assert np.all((mp > 0) & (mp <= 1.0 + 1e-6))
    # the plain call (no max_prob) gives bit-identical outputs
    plain = _blasst().attn_fwd(qd, kd, vd, factor, want_mask=True)
    torch.cuda.synchronize()
    assert torch.equal(plain.o, res.o) and torch.equal(plain.lse, res.lse)


def _packed(lengths_q, lengths_k, H=3, seed=5):
    """Packed documents: token-line clustered Q/K per document, concatenated."""
    qs, ks, vs = [], [], []
    for i, (lq, lk) in enumerate(zip(lengths_q, lengths_k)):
        if lq == 0 and lk == 0:
            continue
        q, k, v = parity.clustered_inputs(1, H, max(lq, 1), max(lk, 1), seed=seed + i)
        qs.append(q[0, :lq])
        ks.append(k[0, :lk])
        vs.append(v[0, :lk])
    q = np.ascontiguousarray(np.concatenate(qs, 0))
    k = np.ascontiguousarray(np.concatenate(ks, 0))
    v = np.ascontiguousarray(np.concatenate(vs, 0))
    cq = np.concatenate([[0], np.cumsum(lengths_q)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lengths_k)]).astype(np.int32)
    return q, k, v, cq, ck


def _packed_to_device(q, k, v, cq, ck):
    import torch
    return (parity.to_device(q), parity.to_device(k), parity.to_device(v),
            torch.from_numpy(cq).cuda(), torch.from_numpy(ck).cuda())


def _check_packed_equals_separate(lq, lk, factor, H=3, seed=5):
    """Each document of a packed call equals the same document alone (bit for bit when the
    decisions agree; lambda rounds differently through the float factor, so otherwise only
    tiles within the decision margin may differ). Documents without keys return O = 0 and
    lse = -inf; documents without queries write nothing."""
    import torch
    q, k, v, cq, ck = _packed(lq, lk, H=H, seed=seed)
    qd, kd, vd, cqd, ckd = _packed_to_device(q, k, v, cq, ck)
    mq, mk = max(max(lq), 1), max(max(lk), 1)
    res = _blasst().attn_varlen_fwd(qd, kd, vd, cqd, ckd, mq, mk, factor, want_max_prob=True)
    torch.cuda.synchronize()
    assert _clear_error() == 0
    counts = res.skip_counts.cpu().numpy().reshape(len(lq), H)
    for i, (a, b_) in enumerate(zip(lq, lk)):
        if a == 0:
            continue
        if b_ == 0:
            assert torch.count_nonzero(res.o[cq[i]:cq[i + 1]]) == 0
            assert torch.all(torch.isinf(res.lse[:, cq[i]:cq[i + 1]]))
            continue
        # the same document alone, with the factor that gives the same lambda = factor / max_seqlen_k
        fd = factor * b_ / mk
        qi, ki, vi = (t[None, s:e].contiguous() for t, s, e in ((qd, cq[i], cq[i + 1]), (kd, ck[i], ck[i + 1]), (vd, ck[i], ck[i + 1])))
        one = _blasst().attn_fwd(qi, ki, vi, fd, want_mask=True, want_max_prob=True)
        torch.cuda.synchronize()
        c1 = one.skip_counts.cpu().numpy()
        if np.array_equal(c1, counts[i]):
            assert torch.equal(one.o[0], res.o[cq[i]:cq[i + 1]])
            assert torch.equal(one.lse[0], res.lse[:, cq[i]:cq[i + 1]])
            assert torch.equal(one.max_prob[0], res.max_prob[:, cq[i]:cq[i + 1]])
        else:
            m1 = one.skip_mask.cpu().numpy()
            ref = oracle.skip_softmax_attn(q[None, cq[i]:cq[i + 1]].copy(), k[None, ck[i]:ck[i + 1]].copy(),
                                           v[None, ck[i]:ck[i + 1]].copy(), 1 / math.sqrt(128), fd)
            gap = ref["gap"].reshape(m1.shape)
            lnlam = math.log(fd / b_) if fd > 0 else -math.inf
            assert np.all(np.abs(gap[m1.astype(bool) != (gap < lnlam)] - lnlam) < parity.MARGIN)
    return counts


@pytest.mark.parametrize("factor", [0.0, 4.0, 64.0])
def test_packed_documents_equal_separate_calls(factor):
    counts = _check_packed_equals_separate([1000, 37, 2048, 300, 129, 1], [1000, 37, 2048, 300, 129, 1], factor)
    if factor > 0:
        assert counts.sum() > 0


@pytest.mark.parametrize("seed", range(6))
def test_random_packed_documents(seed):
    """Seeded random documents: 2 to 6 of them, lengths 0 ... 2100 (some empty, some of one
    token), queries and keys of different lengths, 1 to 4 heads, a random factor."""
    rng = np.random.default_rng(500 + seed)
    n = int(rng.integers(2, 7))
    lq = [int(x) for x in rng.choice([0, 1, 37, 128, 129, 700, 2100], size=n)]
    lk = [int(x) if rng.random() < 0.5 else lq[i] for i, x in enumerate(rng.integers(0, 2100, size=n))]
    lk = [max(x, 1) if lq[i] == 0 else x for i, x in enumerate(lk)]  # (a document needs queries or keys)
    if sum(lq) == 0:
        lq[0] = 64
    if sum(lk) == 0:
        lk[0] = 64
    H = int(rng.integers(1, 5))
    factor = float(rng.choice([0.0, 1.0, 8.0, 64.0]))
    print(lq, lk, H, factor)
    _check_packed_equals_separate(lq, lk, factor, H=H, seed=seed)


def test_packed_documents_against_oracle():
    """Packed documents against the oracle under the full parity bar (max-abs, mean-abs, lse and
    the decision margin rule). A document's decisions in the packed call are those of the same
    document run alone at the same lambda: its outputs must then equal the packed call's bit for
    bit, and the oracle replays that run's skip mask. (If lambda rounds differently through the
    float factor and a decision flips, the flipped tiles must lie within the margin.)"""
    import torch
    lq = [700, 1500, 260]
    lk = [900, 1500, 130]   # cross lengths: queries and keys differ per document
    H = 2
    q, k, v, cq, ck = _packed(lq, lk, H=H, seed=9)
    qd, kd, vd, cqd, ckd = _packed_to_device(q, k, v, cq, ck)
    factor = 8.0
    res = _blasst().attn_varlen_fwd(qd, kd, vd, cqd, ckd, max(lq), max(lk), factor)
    torch.cuda.synchronize()
    assert _clear_error() == 0
    o = res.o.float().cpu().numpy()
    lse = res.lse.cpu().numpy()
    counts = res.skip_counts.cpu().numpy().reshape(len(lq), H)
    replayed = 0
    for i in range(len(lq)):
        sq, eq, sk, ek = cq[i], cq[i + 1], ck[i], ck[i + 1]
        qi, ki, vi = (np.ascontiguousarray(a[None, s:e]) for a, s, e in ((q, sq, eq), (k, sk, ek), (v, sk, ek)))
        fd = factor * lk[i] / max(lk)   # the same lambda = factor / max_seqlen_k
        one = _blasst().attn_fwd(qd[None, sq:eq].contiguous(), kd[None, sk:ek].contiguous(),
                                 vd[None, sk:ek].contiguous(), fd, want_mask=True)
        torch.cuda.synchronize()
        m1 = one.skip_mask.cpu().numpy()
        o_doc = o[None, sq:eq]
        lse_doc = lse[None, :, sq:eq]
        units = parity.sample_units(1, H, lq[i], heads=range(H), qtiles=range(-(-lq[i] // 128)))
        if np.array_equal(one.skip_counts.cpu().numpy(), counts[i]):
            assert torch.equal(one.o[0], res.o[sq:eq]) and torch.equal(one.lse[0], res.lse[:, sq:eq])
            st = parity.compare_units(qi, ki, vi, o_doc, lse_doc, m1, fd, units)
            replayed += 1
            print("document", i, st)
        else:
            ref = oracle.skip_softmax_attn(qi, ki, vi, 1 / math.sqrt(128), fd, units=units,
                                           threads=parity.host_threads())
            gap = ref["gap"].reshape(m1.shape)
            lnlam = math.log(fd / lk[i])
            near = np.abs(gap - lnlam) < parity.MARGIN
            assert np.all(near[m1.astype(bool) != (gap < lnlam)])
            assert np.all(np.abs(counts[i] - m1.reshape(H, -1).sum(-1)) <= near.reshape(H, -1).sum(-1))
    assert replayed >= 2
    assert counts.sum() > 0


def test_min_seq_len_runs_short_documents_dense():
    import torch
    lq = lk = [300, 1200, 100]
    q, k, v, cq, ck = _packed(lq, lk, H=2, seed=21)
    qd, kd, vd, cqd, ckd = _packed_to_device(q, k, v, cq, ck)
    res = _blasst().attn_varlen_fwd(qd, kd, vd, cqd, ckd, 1200, 1200, 64.0, min_seq_len=301)
    torch.cuda.synchronize()
    counts = res.skip_counts.cpu().numpy().reshape(3, 2)
    assert counts[0].sum() == 0 and counts[2].sum() == 0
    for i in (0, 2):
        qi, ki, vi = (t[None, s:e].contiguous() for t, s, e in ((qd, cq[i], cq[i + 1]), (kd, ck[i], ck[i + 1]), (vd, ck[i], ck[i + 1])))
        dense = _blasst().attn_fwd(qi, ki, vi, 0.0)
        torch.cuda.synchronize()
        assert torch.equal(dense.o[0], res.o[cq[i]:cq[i + 1]])


def test_document_without_keys_and_without_queries():
    import torch
    lq = [200, 0, 150, 64]
    lk = [200, 90, 0, 64]
    q, k, v, cq, ck = _packed(lq, lk, H=2, seed=3)
    qd, kd, vd, cqd, ckd = _packed_to_device(q, k, v, cq, ck)
    res = _blasst().attn_varlen_fwd(qd, kd, vd, cqd, ckd, 200, 200, 4.0, want_max_prob=True)
    torch.cuda.synchronize()
    assert _clear_error() == 0
    s, e = cq[2], cq[3]  # document 2 has queries but no keys
    assert torch.count_nonzero(res.o[s:e]) == 0
    assert torch.all(torch.isinf(res.lse[:, s:e]) & (res.lse[:, s:e] < 0))
    assert torch.all(res.max_prob[:, s:e] == 0)
    assert torch.all(torch.isfinite(res.lse[:, cq[3]:cq[4]]))


def test_bad_offset_table_is_clamped_and_reported():
    import torch
    lq = lk = [256, 256]
    q, k, v, cq, ck = _packed(lq, lk, H=1, seed=4)
    qd, kd, vd, _, _ = _packed_to_device(q, k, v, cq, ck)
    bad_q = torch.tensor([0, 300, 200], dtype=torch.int32, device="cuda")   # out of order, past max
    bad_k = torch.tensor([0, 256, 9999], dtype=torch.int32, device="cuda")  # past the tensor
    _clear_error()
    _blasst().attn_varlen_fwd(qd, kd, vd, bad_q, bad_k, 256, 256, 2.0)
    torch.cuda.synchronize()
    st, word = _blasst().blasst_device_error(clear=True)
    assert word & (1 << 4)
    # the context is still usable
    ok = _blasst().attn_varlen_fwd(qd, kd, vd, torch.from_numpy(cq).cuda(), torch.from_numpy(ck).cuda(), 256, 256, 2.0)
    torch.cuda.synchronize()
    assert _clear_error() == 0
    assert torch.isfinite(ok.o.float()).all()
