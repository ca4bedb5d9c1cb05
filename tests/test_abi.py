"""The C ABI without a GPU: the library builds and loads, exports every call
include/specverify.h declares, and rejects bad arguments on the host before
touching the device."""

import ctypes
import os
import re

import pytest

from speculative_decoding_verification_47_gb300 import binding as sb
from speculative_decoding_verification_47_gb300 import build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return sb.lib()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_call(lib):
    names = header_functions()
    assert "sv_spec_verify" in names and "sv_kv_commit" in names
    assert "sv_lmhead_rmsnorm" in names and "sv_spec_verify_noalloc" in names
    for n in names:
        assert hasattr(lib, n), n
    assert sb.sv_version() >= 100


def test_workspace_size(lib):
    assert sb.sv_workspace_size(256, 8, 128256, sb.SV_BF16) > 256 + 256 * 8
    assert sb.sv_workspace_size(0, 8, 10, sb.SV_BF16) == 0
    assert sb.sv_workspace_size(4, 21, 10, sb.SV_BF16) == 0
    assert sb.sv_workspace_size(4, 2, 10, 7) == 0
    a = sb.sv_workspace_size(8, 4, 100, sb.SV_F32)
    assert a % 256 == 0 and a == sb.sv_workspace_size(8, 4, 10**6, sb.SV_BF16)


P = 1 << 20  # an aligned dummy address; none of these calls reaches the device


def _verify(**kw):
    a = dict(target=P, ts=0, tp=0, draft=P, ds=0, dp=0, dtype=sb.SV_BF16, B=4, K=3, V=100,
             tokens=P, kpr=None, temp=None, top_p=1.0, unif=P, mode=None, out=P, n=P, diag=None,
             ws=P, wsb=1 << 30)
    a.update(kw)
    sb.sv_spec_verify(a["target"], a["ts"], a["tp"], a["draft"], a["ds"], a["dp"], a["dtype"],
                      a["B"], a["K"], a["V"], a["tokens"], a["kpr"], a["temp"], a["top_p"],
                      a["unif"], a["mode"], a["out"], a["n"], a["diag"], a["ws"], a["wsb"], 0)


@pytest.mark.parametrize("kw,status", [
    (dict(dtype=5), sb.SV_ERR_DTYPE),
    (dict(B=0), sb.SV_ERR_SHAPE),
    (dict(K=21), sb.SV_ERR_SHAPE),
    (dict(V=0), sb.SV_ERR_SHAPE),
    (dict(target=None), sb.SV_ERR_ARG),
    (dict(unif=None), sb.SV_ERR_ARG),
    (dict(out=None), sb.SV_ERR_ARG),
    (dict(tokens=None), sb.SV_ERR_ARG),
    (dict(draft=None), sb.SV_ERR_ARG),
    (dict(top_p=0.0), sb.SV_ERR_ARG),
    (dict(top_p=1.5), sb.SV_ERR_ARG),
    (dict(target=P + 1), sb.SV_ERR_ARG),
    (dict(tp=50), sb.SV_ERR_SHAPE),
    (dict(ts=-1), sb.SV_ERR_SHAPE),
    (dict(ws=None), sb.SV_ERR_WORKSPACE),
    (dict(ws=P + 16), sb.SV_ERR_WORKSPACE),
    (dict(wsb=16), sb.SV_ERR_WORKSPACE),
    (dict(B=(1 << 27) // 21 + 1, K=20), sb.SV_ERR_SHAPE),  # grid of B*(K+1) clusters
])
def test_spec_verify_host_checks(lib, kw, status):
    with pytest.raises(sb.SVError) as e:
        _verify(**kw)
    assert e.value.status == status
    assert sb.sv_last_error()


def test_kv_commit_and_lmhead_host_checks(lib):
    with pytest.raises(sb.SVError) as e:
        sb.sv_kv_commit(None, P, None, None, 4, 3, P, 256, 0)
    assert e.value.status == sb.SV_ERR_ARG
    with pytest.raises(sb.SVError) as e:
        sb.sv_kv_commit(P, P, None, None, 4, 3, P + 8, 256, 0)
    assert e.value.status == sb.SV_ERR_WORKSPACE
    with pytest.raises(sb.SVError) as e:
        sb.sv_lmhead_rmsnorm(P, P, 1e-5, P, P, sb.SV_BF16, 4, 100, 128, P, 1 << 30, 0)
    assert e.value.status == sb.SV_ERR_SHAPE
    with pytest.raises(sb.SVError) as e:
        sb.sv_lmhead_rmsnorm(P, P, 1e-5, P, P, 9, 4, 128, 128, P, 1 << 30, 0)
    assert e.value.status == sb.SV_ERR_DTYPE


def test_noalloc_host_checks(lib):
    with pytest.raises(sb.SVError) as e:
        sb.sv_spec_verify_noalloc(P, 0, 0, P, 0, 0, sb.SV_BF16, 8192, 20, 32000, P, None, None,
                                  1.0, P, None, P, P, None, 0)
    assert e.value.status == sb.SV_ERR_WORKSPACE
    with pytest.raises(sb.SVError) as e:
        sb.sv_spec_verify_noalloc(None, 0, 0, P, 0, 0, sb.SV_BF16, 4, 3, 100, P, None, None,
                                  1.0, P, None, P, P, None, 0)
    assert e.value.status == sb.SV_ERR_ARG


def test_draft_sample_host_checks(lib):
    assert "sv_draft_sample" in header_functions()
    assert sb.sv_draft_sample_workspace_size() == 256

    def call(**kw):
        a = dict(logits=P, ss=0, ps=0, dtype=sb.SV_BF16, B=4, K=3, V=100, kpr=None, temp=None,
                 top_p=1.0, unif=P, mode=None, out=P, ws=P, wsb=256)
        a.update(kw)
        sb.sv_draft_sample(a["logits"], a["ss"], a["ps"], a["dtype"], a["B"], a["K"], a["V"],
                           a["kpr"], a["temp"], a["top_p"], a["unif"], a["mode"], a["out"],
                           a["ws"], a["wsb"], 0)

    for kw, status in [(dict(dtype=5), sb.SV_ERR_DTYPE), (dict(B=0), sb.SV_ERR_SHAPE),
                       (dict(K=0), sb.SV_ERR_SHAPE), (dict(logits=None), sb.SV_ERR_ARG),
                       (dict(unif=None), sb.SV_ERR_ARG), (dict(top_p=0.0), sb.SV_ERR_ARG),
                       (dict(logits=P + 1), sb.SV_ERR_ARG), (dict(ps=50), sb.SV_ERR_SHAPE),
                       (dict(ws=None), sb.SV_ERR_WORKSPACE), (dict(wsb=255), sb.SV_ERR_WORKSPACE)]:
        with pytest.raises(sb.SVError) as e:
            call(**kw)
        assert e.value.status == status, kw


def test_dynk_host_checks(lib):
    assert sb.sv_dynk_state_size(0) == 0
    assert sb.sv_dynk_state_size(256) >= 256 * (7 * 4 + 128)
    with pytest.raises(sb.SVError) as e:
        sb.sv_dynk_init(P, 0, 4, 0)
    assert e.value.status == sb.SV_ERR_SHAPE
    with pytest.raises(sb.SVError) as e:
        sb.sv_dynk_init(None, 4, 4, 0)
    assert e.value.status == sb.SV_ERR_ARG
    with pytest.raises(sb.SVError) as e:
        sb.sv_dynk_update(P, 4, None, P, None, P, P, 256, 0)
    assert e.value.status == sb.SV_ERR_ARG
    with pytest.raises(sb.SVError) as e:
        sb.sv_dynk_update(P, 4, P, P, None, P, None, 256, 0)
    assert e.value.status == sb.SV_ERR_WORKSPACE


def test_kv_commit_paged_host_checks(lib):
    with pytest.raises(sb.SVError) as e:
        sb.sv_kv_commit_paged(P, P, P, P, 0, 16, P, P, 10, 4, P, 256, 0)
    assert e.value.status == sb.SV_ERR_SHAPE
    with pytest.raises(sb.SVError) as e:
        sb.sv_kv_commit_paged(P, P, None, P, 4, 16, P, P, 10, 4, P, 256, 0)
    assert e.value.status == sb.SV_ERR_ARG
    with pytest.raises(sb.SVError) as e:
        sb.sv_kv_commit_paged(P, P, P, P, 4, 16, P, P, 10, 4, P, 8, 0)
    assert e.value.status == sb.SV_ERR_WORKSPACE
    # lengths are int32 on the device: a full table plus one page must fit
    with pytest.raises(sb.SVError) as e:
        sb.sv_kv_commit_paged(P, P, P, P, (1 << 31) // 16 - 1, 16, P, P, 10, 4, P, 256, 0)
    assert e.value.status == sb.SV_ERR_SHAPE
    with pytest.raises(sb.SVError) as e:
        sb.sv_kv_commit_paged(P, P, P, P, 4, 16, P, P, 10, (1 << 30) + 1, P, 256, 0)
    assert e.value.status == sb.SV_ERR_SHAPE


def test_sequence_count_limits(lib):
    assert sb.sv_dynk_state_size((1 << 30) + 1) == 0
    with pytest.raises(sb.SVError) as e:
        sb.sv_dynk_init(P, (1 << 30) + 1, 4, 0)
    assert e.value.status == sb.SV_ERR_SHAPE
    with pytest.raises(sb.SVError) as e:
        sb.sv_kv_commit(P, P, None, None, (1 << 30) + 1, 3, P, 256, 0)
    assert e.value.status == sb.SV_ERR_SHAPE
    with pytest.raises(sb.SVError) as e:
        sb.sv_draft_sample(P, 0, 0, sb.SV_BF16, (1 << 27) // 8 + 1, 8, 100, None, None, 1.0, P,
                           None, P, P, 256, 0)
    assert e.value.status == sb.SV_ERR_SHAPE


def test_host_tensors_are_refused(lib):
    """A host tensor never reaches a device-pointer argument."""
    import torch
    host = torch.zeros(16, dtype=torch.int32)
    with pytest.raises(ValueError):
        sb.sv_kv_commit(host, P, None, None, 4, 3, P, 256, 0)
    with pytest.raises(ValueError):
        sb.sv_read_device_flags(host.pin_memory() if torch.cuda.is_available() else host, 0)


def test_noalloc_limits_match_the_header(lib):
    """The header's examples of batches the allocation-free call accepts
    (workspace <= 2 MiB) and refuses, checked on sv_workspace_size."""
    cap = 2 << 20
    for B, K in [(4096, 20), (8192, 14), (16384, 6)]:
        assert sb.sv_workspace_size(B, K, 128256, sb.SV_BF16) <= cap, (B, K)
    for B, K in [(8192, 15), (16384, 7)]:
        assert sb.sv_workspace_size(B, K, 128256, sb.SV_BF16) > cap, (B, K)
