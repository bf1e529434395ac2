"""The C ABI without a GPU: the library loads, exports every entry point the
header declares, and rejects bad arguments on the host before any CUDA call."""
import os
import re

import pytest

from vocab_embedding_cross_gb300 import _lib as vce

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(vce.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return vce.lib()


def declared_functions():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^\s*[a-z_0-9]+\**\s+\**(vce_[a-z_0-9]+)\s*\(", src, re.M))
    return sorted(names)


def test_every_declared_symbol_exported(L):
    names = declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for s in range(7):
        assert vce.status_str(s).startswith("VCE_")
    assert vce.vce_embed_bwd_chunk() == 32
    assert vce.vce_version() >= 100


def P(**kw):
    base = dict(T=64, H=64, Vp=1024, V_real=1000, S=4, dtype=vce.VCE_BF16)
    base.update(kw)
    return vce.problem(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(Vp=1000), vce.VCE_ERR_ARG),            # not a multiple of 64
    (dict(Vp=0), vce.VCE_ERR_ARG),
    (dict(V_real=1025), vce.VCE_ERR_ARG),
    (dict(V_real=0), vce.VCE_ERR_ARG),
    (dict(S=0), vce.VCE_ERR_ARG),
    (dict(S=1025), vce.VCE_ERR_ARG),
    (dict(T=-1), vce.VCE_ERR_ARG),
    (dict(H=0), vce.VCE_ERR_ARG),
    (dict(H=4), vce.VCE_ERR_UNSUPPORTED),         # 8 bytes per bf16 row
    (dict(dtype=7), vce.VCE_ERR_UNSUPPORTED),
    (dict(T=1 << 31), vce.VCE_ERR_UNSUPPORTED),
    (dict(T=(1 << 31) - 1, Vp=1 << 30, V_real=1 << 30), vce.VCE_ERR_UNSUPPORTED),   # 2^41 work items
    (dict(ignore_index=0), vce.VCE_ERR_ARG),     # the ignore value names a real class
    (dict(ignore_index=999), vce.VCE_ERR_ARG),
    (dict(flags=4), vce.VCE_ERR_ARG),            # no such flag
    (dict(flags=1 << 20), vce.VCE_ERR_ARG),
])
def test_bad_problem_rejected_on_host(L, kw, code):
    p = P(**kw)
    assert vce.vce_workspace_size(p, vce.VCE_OP_LOSS_FWD) == vce.SIZE_MAX
    for fn, args in ((L.vce_embed_fwd, (None,) * 7), (L.vce_embed_bwd, (None, None, None, None, 0, None, None)),
                     (L.vce_embed_bwd_plan, (None, None, 0, None, None)),
                     (L.vce_embed_fwd_plan, (None,) * 6 + (0, None, None)),
                     (L.vce_embed_bwd_apply, (None, None, None, 0, None, None)),
                     (L.vce_loss_fwd, (None,) * 9 + (0, None, None)),
                     (L.vce_loss_bwd, (None, None, None, None, 1.0, None, None, None, 0, None, None))):
        import ctypes
        assert fn(ctypes.byref(p), *args) == code


def test_null_pointers_rejected(L):
    import ctypes
    p = P()
    assert L.vce_embed_fwd(ctypes.byref(p), None, None, None, None, None, None, None) == vce.VCE_ERR_ARG
    assert L.vce_loss_fwd(ctypes.byref(p), None, None, None, None, None, None, None, None, None, 0, None,
                          None) == vce.VCE_ERR_ARG
    assert L.vce_wait_selftest(1000, None, None) == vce.VCE_ERR_ARG
    assert L.vce_embed_bwd_plan(ctypes.byref(p), None, 0x4000, 1 << 30, None, None) == vce.VCE_ERR_ARG
    assert L.vce_embed_bwd_apply(ctypes.byref(p), None, 0x2000, 0x4000, 1 << 30, None, None) == vce.VCE_ERR_ARG
    assert L.vce_embed_bwd_apply(ctypes.byref(p), 0x2000, None, 0x4000, 1 << 30, None, None) == vce.VCE_ERR_ARG
    assert L.vce_ngram_embed_bwd_plan(ctypes.byref(p), None, 64, 64, 0, 0x4000, 1 << 30, None, None) == \
        vce.VCE_ERR_ARG
    assert L.vce_ngram_embed_bwd_plan(ctypes.byref(p), 0x1000, -1, 64, 0, 0x4000, 1 << 30, None, None) == \
        vce.VCE_ERR_ARG
    assert L.vce_ngram_embed_bwd_plan(ctypes.byref(p), 0x1000, 64, 64, -1, 0x4000, 1 << 30, None, None) == \
        vce.VCE_ERR_ARG                            # negative sequence length
    assert L.vce_ngram_embed_bwd_apply(ctypes.byref(p), 0x2000, 0x3000, None, 64, None, 0, 0x4000, 1 << 30,
                                       None, None) == vce.VCE_ERR_ARG   # a 2-gram table without its gradient
    assert L.vce_ngram_embed_bwd_apply(ctypes.byref(p), None, 0x3000, None, 0, None, 0, 0x4000, 1 << 30,
                                       None, None) == vce.VCE_ERR_ARG
    # an empty batch has nothing to plan or apply
    p0 = P(T=0)
    assert L.vce_embed_bwd_plan(ctypes.byref(p0), None, None, 0, None, None) == vce.VCE_OK
    assert L.vce_embed_bwd_apply(ctypes.byref(p0), None, None, None, 0, None, None) == vce.VCE_OK


def test_misaligned_pointers_rejected(L):
    import ctypes
    p = P()
    # 8-byte aligned but not 16-byte aligned matrices; never dereferenced
    assert L.vce_embed_fwd(ctypes.byref(p), 0x1000, 0x1008, 0x2000, None, None, None, None) == \
        vce.VCE_ERR_UNSUPPORTED


def test_workspace_sizes(L):
    p = P(T=8192, H=2048, Vp=151936, V_real=151936, S=8)
    assert vce.vce_workspace_size(p, vce.VCE_OP_EMBED_FWD) == 0
    fwd = vce.vce_workspace_size(p, vce.VCE_OP_LOSS_FWD)
    units = 8 * -(-(151936 // 8) // 2048)
    assert fwd >= 8192 * units * 8 + 8192 * 4
    mn = vce.vce_workspace_size_min(p, vce.VCE_OP_LOSS_BWD)
    rec = vce.vce_workspace_size(p, vce.VCE_OP_LOSS_BWD)
    assert mn == 256 + 8192 * 256 * 2 and rec > mn
    assert vce.vce_workspace_size(p, vce.VCE_OP_EMBED_BWD) > 8192 * 16
    # the embedding backward workspace holds keys, runs and run partial slots
    p4 = P(T=16384, H=3072, Vp=201088, V_real=201088, S=8)
    assert vce.vce_workspace_size(p4, vce.VCE_OP_EMBED_BWD) < 64 << 20


def test_bf16_dh_workspace(L):
    """A bf16 dH adds its fp32 sum (T*H*4 bytes) to both backward sizes, and a
    workspace without room for it is refused before anything is launched."""
    import ctypes
    for T, H in ((8192, 2048), (100, 72)):
        p = P(T=T, H=H, Vp=151936, V_real=151936, S=8)
        q = P(T=T, H=H, Vp=151936, V_real=151936, S=8, flags=vce.VCE_FLAG_DH_BF16)
        acc = -(-(T * H * 4) // 256) * 256
        for fn in (vce.vce_workspace_size, vce.vce_workspace_size_min):
            assert fn(q, vce.VCE_OP_LOSS_BWD) == fn(p, vce.VCE_OP_LOSS_BWD) + acc
        both = P(T=T, H=H, Vp=151936, V_real=151936, S=8,
                 flags=vce.VCE_FLAG_DH_BF16 | vce.VCE_FLAG_ACCUMULATE_DH)
        assert vce.vce_workspace_size(both, vce.VCE_OP_LOSS_BWD) == vce.vce_workspace_size(q, vce.VCE_OP_LOSS_BWD)
        mn = vce.vce_workspace_size_min(q, vce.VCE_OP_LOSS_BWD)
        args = (0x1000, 0x2000, 0x3000, 0x4000, 1.0, 0x5000, 0x6000, 0x10000)
        assert L.vce_loss_bwd(ctypes.byref(q), *args, mn - 256, None, None) == vce.VCE_ERR_WORKSPACE
        assert L.vce_loss_bwd(ctypes.byref(q), *args, acc - 256, None, None) == vce.VCE_ERR_WORKSPACE
    # the sampled loss's workspace holds the sum too
    q = P(T=4096, H=1024, Vp=50048, V_real=50000, S=8, flags=vce.VCE_FLAG_DH_BF16)
    p = P(T=4096, H=1024, Vp=50048, V_real=50000, S=8)
    assert vce.vce_sampled_workspace_size(q, 8192) >= vce.vce_sampled_workspace_size(p, 8192) + 4096 * 1024 * 4


def test_workspace_too_small_rejected_on_host(L):
    import ctypes
    p = P(T=64)
    need = vce.vce_workspace_size(p, vce.VCE_OP_EMBED_BWD)
    assert L.vce_embed_bwd(ctypes.byref(p), 0x1000, 0x2000, 0x3000, 0x4000, need - 1, None, None) == \
        vce.VCE_ERR_WORKSPACE
    assert L.vce_embed_bwd(ctypes.byref(p), 0x1000, 0x2000, 0x3000, 0x4010, need, None, None) == \
        vce.VCE_ERR_WORKSPACE                      # misaligned workspace
    # the plan and its application use the same workspace size and alignment
    assert L.vce_embed_fwd_plan(ctypes.byref(p), 0x1000, 0x2000, 0x3000, None, None, 0x4000, need - 1, None,
                                None) == vce.VCE_ERR_WORKSPACE
    assert L.vce_embed_fwd_plan(ctypes.byref(p), 0x1000, 0x2008, 0x3000, None, None, 0x4000, need, None,
                                None) == vce.VCE_ERR_UNSUPPORTED   # W not 16-byte aligned
    assert L.vce_embed_fwd_plan(ctypes.byref(p), 0x1000, None, 0x3000, None, None, 0x4000, need, None,
                                None) == vce.VCE_ERR_ARG
    assert L.vce_embed_bwd_plan(ctypes.byref(p), 0x1000, 0x4000, need - 1, None, None) == vce.VCE_ERR_WORKSPACE
    assert L.vce_embed_bwd_plan(ctypes.byref(p), 0x1000, 0x4010, need, None, None) == vce.VCE_ERR_WORKSPACE
    assert L.vce_embed_bwd_plan(ctypes.byref(p), 0x1000, None, need, None, None) == vce.VCE_ERR_WORKSPACE
    assert L.vce_embed_bwd_apply(ctypes.byref(p), 0x2000, 0x3000, 0x4000, need - 1, None, None) == \
        vce.VCE_ERR_WORKSPACE
    assert L.vce_embed_bwd_apply(ctypes.byref(p), 0x2000, 0x3000, None, need, None, None) == vce.VCE_ERR_WORKSPACE
    assert L.vce_embed_bwd_apply(ctypes.byref(p), 0x2008, 0x3000, 0x4000, need, None, None) == \
        vce.VCE_ERR_UNSUPPORTED                    # dE not 16-byte aligned
    ng = vce.vce_ngram_workspace_size(p)
    assert L.vce_ngram_embed_bwd_plan(ctypes.byref(p), 0x1000, 64, 64, 0, 0x4000, ng - 1, None, None) == \
        vce.VCE_ERR_WORKSPACE
    assert L.vce_ngram_embed_bwd_apply(ctypes.byref(p), 0x2000, 0x3000, 0x5000, 64, 0x6000, 64, 0x4010, ng,
                                       None, None) == vce.VCE_ERR_WORKSPACE


def test_sampled_candidates_rejected_on_host(L):
    import ctypes
    p = P(dtype=vce.VCE_F32)
    ws_need = vce.vce_workspace_size(p, vce.VCE_OP_SAMPLED_CANDIDATES)
    assert 2 * 4 * ((1000 + 31) // 32) <= ws_need < vce.SIZE_MAX   # bitmap and word prefixes
    fake = 1 << 20   # never dereferenced: every case below fails validation first
    call = L.vce_sampled_candidates
    assert call(ctypes.byref(p), fake, fake, 10, 0, fake, fake, fake, fake, ws_need, None, None) == vce.VCE_ERR_ARG
    assert call(ctypes.byref(p), fake, fake, 10, 1001, fake, fake, fake, fake, ws_need, None,
                None) == vce.VCE_ERR_ARG
    assert call(ctypes.byref(p), None, fake, 10, 100, fake, fake, fake, fake, ws_need, None,
                None) == vce.VCE_ERR_ARG
    assert call(ctypes.byref(p), fake, fake, 10, 100, fake, fake, fake, fake, ws_need - 1, None,
                None) == vce.VCE_ERR_WORKSPACE
    assert call(ctypes.byref(p), fake, fake, 10, 100, fake, fake, fake, None, ws_need, None,
                None) == vce.VCE_ERR_WORKSPACE


def test_ignore_value_outside_the_real_classes_accepted(L):
    """-100, V_real and any value past the padded vocabulary are all usable
    ignore values: only one naming a real class is refused."""
    for ig in (-100, -1, 1000, 1023, 5000):
        assert vce.vce_workspace_size(P(ignore_index=ig), vce.VCE_OP_LOSS_FWD) != vce.SIZE_MAX


def test_noalloc_checks_like_the_workspace_forward(L):
    """The allocation-free forward applies vce_loss_fwd's argument rules: the
    same problems are refused with the same codes, and the bf16-dH flag that a
    caller may share between forward and backward is accepted by both."""
    import ctypes
    fake = 1 << 20   # never dereferenced: every case below fails validation first
    for kw, code in ((dict(Vp=1000), vce.VCE_ERR_ARG), (dict(flags=4), vce.VCE_ERR_ARG),
                     (dict(ignore_index=0), vce.VCE_ERR_ARG), (dict(H=4), vce.VCE_ERR_UNSUPPORTED),
                     (dict(T=(1 << 31) - 1, Vp=1 << 30, V_real=1 << 30), vce.VCE_ERR_UNSUPPORTED)):
        p = P(**kw)
        a = L.vce_loss_fwd(ctypes.byref(p), fake, fake, fake, fake, fake, None, None, None, fake, 1 << 30, None,
                           None)
        b = L.vce_loss_fwd_noalloc(ctypes.byref(p), fake, fake, fake, fake, fake, None, None, None, None, None)
        assert a == b == code, (kw, a, b)
    # the flags vce_loss_fwd accepts pass the noalloc check too: the call gets as
    # far as the alignment check of h (8-byte aligned here, 16 needed)
    for flags in (vce.VCE_FLAG_DH_BF16, vce.VCE_FLAG_ACCUMULATE_DH | vce.VCE_FLAG_DH_BF16):
        p = P(flags=flags)
        assert L.vce_loss_fwd_noalloc(ctypes.byref(p), fake + 8, fake, fake, fake, fake, None, None, None, None,
                                      None) == vce.VCE_ERR_UNSUPPORTED
        assert vce.vce_workspace_size(p, vce.VCE_OP_LOSS_FWD) != vce.SIZE_MAX
