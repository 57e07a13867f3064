"""The C ABI without a GPU: the library loads, exports every function that
include/dsa.h declares, and rejects invalid host arguments before touching
the device (no compute call is made here)."""
import ctypes

import pytest

import __graft_entry__  # noqa: F401  (puts the repo root on sys.path)
from sparse_attention_gemm_gb300 import build as dsa_build
from sparse_attention_gemm_gb300 import ops


@pytest.fixture(scope="module")
def lib():
    dsa_build.build()
    return ops.lib()


def test_header_declares_the_hot_path():
    names = ops.header_functions()
    for must in ["dsa_thd_metadata", "dsa_indexer_scores", "dsa_topk", "dsa_compact_sort_indices",
                 "dsa_indexer_topk_workspace_size", "dsa_indexer_topk", "dsa_indexer_topk_ex", "dsa_topk_softmax",
                 "dsa_sparse_attn_fwd", "dsa_sparse_attn_fwd_ex", "dsa_forward_host",
                 "dsa_pack_routes", "dsa_thd_metadata_ratio", "dsa_indexer_scores_ratio", "dsa_indexer_topk_ratio",
                 "dsa_indexer_scores_fp8", "dsa_indexer_topk_fp8", "dsa_sparse_attn_bwd",
                 "dsa_sparse_attn_bwd_workspace_size", "dsa_sparse_attn_bwd_ex",
                 "dsa_sparse_attn_bwd_workspace_size_ex",
                 "dsa_last_error", "dsa_device_status"]:
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in ops.header_functions():
        assert hasattr(lib, name), name
        assert name in ops._SIGNATURES, f"binding lacks {name}"


NULL = None
FAKE = ctypes.c_void_p(4096)  # never dereferenced: validation fails first


@pytest.mark.parametrize("call", [
    lambda L: L.dsa_thd_metadata(FAKE, 0, 10, FAKE, FAKE, NULL),
    lambda L: L.dsa_thd_metadata(NULL, 1, 10, FAKE, FAKE, NULL),
    lambda L: L.dsa_topk(FAKE, 16, FAKE, NULL, 4, 0, FAKE, NULL, NULL, NULL),
    lambda L: L.dsa_topk(FAKE, 16, FAKE, NULL, 4, 2049, FAKE, NULL, NULL, NULL),
    lambda L: L.dsa_topk(NULL, 16, FAKE, NULL, 4, 8, FAKE, NULL, NULL, NULL),
    lambda L: L.dsa_compact_sort_indices(FAKE, 4, 0, 10, FAKE, FAKE, NULL),
    lambda L: L.dsa_compact_sort_indices(FAKE, 4, 16385, 10, FAKE, FAKE, NULL),
    lambda L: L.dsa_indexer_scores(FAKE, FAKE, FAKE, FAKE, 1, 128, 64, 96, 128, FAKE, 128, NULL),
    lambda L: L.dsa_indexer_scores(FAKE, FAKE, FAKE, FAKE, 1, 128, 48, 128, 128, FAKE, 128, NULL),
    lambda L: L.dsa_indexer_scores(FAKE, FAKE, FAKE, FAKE, 1, 128, 64, 128, 128, FAKE, 126, NULL),
    lambda L: L.dsa_indexer_scores(ctypes.c_void_p(4097), FAKE, FAKE, FAKE, 1, 128, 64, 128, 128, FAKE, 128, NULL),
    lambda L: L.dsa_indexer_topk(FAKE, FAKE, FAKE, FAKE, 1, 128, 64, 128, 0, 128, FAKE, NULL, FAKE, 1 << 30, NULL),
    lambda L: L.dsa_sparse_attn_fwd(FAKE, FAKE, NULL, FAKE, NULL, NULL, 4, 4, 64, 576, 256, 8, 0.1, FAKE, FAKE,
                                    NULL, NULL, NULL),
    lambda L: L.dsa_sparse_attn_fwd(FAKE, FAKE, NULL, FAKE, NULL, NULL, 4, 4, 129, 576, 512, 8, 0.1, FAKE, FAKE,
                                    NULL, NULL, NULL),
    lambda L: L.dsa_sparse_attn_fwd(FAKE, FAKE, NULL, FAKE, NULL, NULL, 4, 4, 64, 576, 512, 8, 0.0, FAKE, FAKE,
                                    NULL, NULL, NULL),
    lambda L: L.dsa_sparse_attn_fwd(FAKE, FAKE, NULL, FAKE, NULL, NULL, 4, 4, 64, 576, 512, 8, float("inf"), FAKE,
                                    FAKE, NULL, NULL, NULL),
    lambda L: L.dsa_sparse_attn_fwd(FAKE, FAKE, NULL, FAKE, NULL, NULL, 4, 4, 64, 256, 256, 8, 0.1, FAKE, FAKE,
                                    NULL, NULL, NULL),
    lambda L: L.dsa_sparse_attn_fwd_ex(FAKE, FAKE, NULL, FAKE, NULL, NULL, 4, 4, 64, 576, 512, 128, 0.1, FAKE, FAKE,
                                       NULL, NULL, 96, FAKE, NULL),
    lambda L: L.dsa_sparse_attn_fwd_ex(FAKE, FAKE, NULL, FAKE, NULL, NULL, 4, 4, 64, 576, 512, 128, 0.1, FAKE, FAKE,
                                       NULL, NULL, 192, FAKE, NULL),
    lambda L: L.dsa_sparse_attn_fwd_ex(FAKE, FAKE, NULL, FAKE, NULL, NULL, 4, 4, 64, 576, 512, 128, 0.1, FAKE, FAKE,
                                       NULL, NULL, 64, NULL, NULL),
    lambda L: L.dsa_topk_softmax(FAKE, FAKE, 4, 0, FAKE, FAKE, NULL),
    lambda L: L.dsa_topk_softmax(FAKE, FAKE, 4, 8, NULL, NULL, NULL),
    lambda L: L.dsa_indexer_topk_ex(FAKE, FAKE, FAKE, FAKE, 1, 128, 64, 128, 64, 128, FAKE, NULL, NULL, NULL, NULL,
                                    FAKE, 1 << 30, NULL),
    lambda L: L.dsa_forward_host(NULL, 1, 128, 64, 128, 64, 128, 64, 576, 512, 0.1, 4, NULL, NULL),
    lambda L: L.dsa_forward_host(ctypes.byref(ops.ForwardBuffers()), 1, 128, 64, 128, 64, 128, 64, 576, 512, 0.1, 0,
                                 NULL, NULL),
    lambda L: L.dsa_forward_host(ctypes.byref(ops.ForwardBuffers()), 1, 128, 64, 128, 64, 128, 64, 576, 512, 0.1, 4,
                                 NULL, NULL),
    lambda L: L.dsa_pack_routes(FAKE, 0, 4, 4, FAKE, NULL),
    lambda L: L.dsa_indexer_candidates(FAKE, FAKE, FAKE, FAKE, 1, 128, 64, 128, 0, 128, FAKE, 1 << 30, NULL),
    lambda L: L.dsa_indexer_candidates(FAKE, FAKE, FAKE, FAKE, 1, 128, 64, 128, 64, 129, FAKE, 1 << 30, NULL),
    lambda L: L.dsa_select_candidates(FAKE, 1, 128, 64, 128, 64, 128, FAKE, 1 << 30, NULL, NULL, NULL),
    lambda L: L.dsa_select_candidates(NULL, 1, 128, 64, 128, 64, 128, FAKE, 1 << 30, FAKE, NULL, NULL),
    lambda L: L.dsa_select_candidates(FAKE, 1, 128, 64, 128, 0, 128, FAKE, 1 << 30, FAKE, NULL, NULL),
    lambda L: L.dsa_indexer_scores_fp8(FAKE, FAKE, NULL, FAKE, FAKE, FAKE, FAKE, NULL, 1, 128, 128, 64, 128, 1, 128,
                                       FAKE, 128, NULL),
    lambda L: L.dsa_indexer_scores_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 1, 128, 128, 64, 64, 1, 128,
                                       FAKE, 128, NULL),
    lambda L: L.dsa_indexer_scores_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 1, 128, 128, 16, 128, 1, 128,
                                       FAKE, 128, NULL),
    lambda L: L.dsa_indexer_topk_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 1, 128, 128, 64, 128, 1, 64, 128,
                                     NULL, NULL, NULL, NULL, NULL, FAKE, 1 << 30, NULL),
    lambda L: L.dsa_sparse_attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, FAKE, NULL, 4, 8, 64, 512, 512, 8, 0.1, FAKE,
                                    FAKE, NULL, FAKE, 1 << 30, NULL),
    lambda L: L.dsa_sparse_attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, FAKE, NULL, 4, 8, 129, 576, 512, 8, 0.1, FAKE,
                                    FAKE, NULL, FAKE, 1 << 30, NULL),
    lambda L: L.dsa_sparse_attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, FAKE, NULL, 4, 8, 64, 576, 512, 8, 0.0, FAKE,
                                    FAKE, NULL, FAKE, 1 << 30, NULL),
    lambda L: L.dsa_sparse_attn_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, FAKE, NULL, 4, 8, 64, 576, 512, 8, 0.1, NULL,
                                    FAKE, NULL, FAKE, 1 << 30, NULL),
    lambda L: L.dsa_sparse_attn_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, FAKE, NULL, 4, 8, 64, 512, 512, 8, 0.1,
                                       FAKE, FAKE, NULL, 0, FAKE, 1 << 30, NULL),
    lambda L: L.dsa_sparse_attn_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, FAKE, NULL, 4, 8, 64, 576, 512, 8, 0.1,
                                       FAKE, NULL, NULL, 0, FAKE, 1 << 30, NULL),
    lambda L: L.dsa_thd_metadata_ratio(FAKE, FAKE, NULL, 1, 10, 0, FAKE, FAKE, NULL),
    lambda L: L.dsa_thd_metadata_ratio(FAKE, NULL, NULL, 1, 10, 4, FAKE, FAKE, NULL),
    lambda L: L.dsa_indexer_scores_ratio(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 1, 128, 32, 64, 128, 0, 32, FAKE, 32, NULL),
    lambda L: L.dsa_indexer_scores_ratio(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 1, 128, 32, 64, 128, 4, 33, FAKE, 36, NULL),
    lambda L: L.dsa_indexer_scores_ratio(FAKE, FAKE, FAKE, FAKE, NULL, NULL, 1, 128, 32, 64, 128, 4, 32, FAKE, 32, NULL),
    lambda L: L.dsa_indexer_scores_ratio(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 1, 128, 0, 64, 128, 4, 1, FAKE, 4, NULL),
    lambda L: L.dsa_indexer_scores_ratio(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 1, 128, 32, 64, 128, 4, 32, FAKE, 30, NULL),
    lambda L: L.dsa_indexer_topk_ratio(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 1, 128, 32, 64, 128, 4, 0, 32, FAKE, NULL,
                                       NULL, NULL, NULL, FAKE, 1 << 30, NULL),
    lambda L: L.dsa_indexer_topk_ratio(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 1, 128, 32, 64, 128, 4, 16, 32, FAKE, NULL,
                                       NULL, FAKE, NULL, FAKE, 1 << 30, NULL),
    lambda L: L.dsa_indexer_topk_ratio(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 1, 128, 32, 64, 128, 4, 16, 32, NULL, NULL,
                                       NULL, NULL, NULL, FAKE, 1 << 30, NULL),
])
def test_invalid_arguments_are_rejected_before_launch(lib, call):
    assert call(lib) == ops.DSA_ERR_VALUE
    assert len(lib.dsa_last_error()) > 0


def test_workspace_errors(lib):
    need = lib.dsa_indexer_topk_workspace_size(4096, 64, 128, 2048, 4096)
    assert need > 0
    assert lib.dsa_indexer_topk_workspace_size(4096, 64, 128, 4096, 4096) == 0
    rc = lib.dsa_indexer_topk(FAKE, FAKE, FAKE, FAKE, 1, 4096, 64, 128, 2048, 4096, FAKE, NULL, FAKE, need - 1, NULL)
    assert rc == ops.DSA_ERR_WORKSPACE
    rc = lib.dsa_indexer_topk(FAKE, FAKE, FAKE, FAKE, 1, 4096, 64, 128, 2048, 4096, FAKE, NULL,
                              ctypes.c_void_p(4096 + 16), need, NULL)
    assert rc == ops.DSA_ERR_WORKSPACE


def test_ratio_call_checks_the_workspace(lib):
    need = lib.dsa_indexer_topk_workspace_size(4096, 64, 128, 512, 1024)
    rc = lib.dsa_indexer_topk_ratio(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, 1, 4096, 1024, 64, 128, 4, 512, 1024, FAKE,
                                    NULL, NULL, NULL, NULL, FAKE, need - 1, NULL)
    assert rc == ops.DSA_ERR_WORKSPACE


def test_stage_calls_check_the_workspace(lib):
    need = lib.dsa_indexer_topk_workspace_size(4096, 64, 128, 2048, 4096)
    rc = lib.dsa_indexer_candidates(FAKE, FAKE, FAKE, FAKE, 1, 4096, 64, 128, 2048, 4096, FAKE, need - 1, NULL)
    assert rc == ops.DSA_ERR_WORKSPACE
    rc = lib.dsa_select_candidates(FAKE, 1, 4096, 64, 128, 2048, 4096, ctypes.c_void_p(4096 + 16), need, FAKE, NULL,
                                   NULL)
    assert rc == ops.DSA_ERR_WORKSPACE


@pytest.mark.parametrize("T,Tkv,H,K", [(100, 300, 64, 256), (7, 5, 128, 64), (65536, 65536, 64, 2048)])
def test_bwd_workspace_layout(lib, T, Tkv, H, K):
    """The backward's workspace: per (token, head) two fp32 statistics and the
    d_sink row term, then scale * dS and P of every slot (bf16, heads padded
    to groups of 64), then, in the deterministic variant only, the 152 fp32
    dkv copies.  Every part starts on a 256-byte boundary."""
    def a256(x):
        return (x + 255) // 256 * 256

    hp = (H + 63) // 64 * 64
    atomic = a256(T * H * 8) + a256(T * H * 4) + 2 * a256(T * K * hp * 2)
    assert lib.dsa_sparse_attn_bwd_workspace_size_ex(T, Tkv, H, K, 0) == atomic
    det = atomic + a256(152 * Tkv * 576 * 4)
    assert lib.dsa_sparse_attn_bwd_workspace_size_ex(T, Tkv, H, K, 1) == det
    assert lib.dsa_sparse_attn_bwd_workspace_size(T, Tkv, H, K) == det


def test_bwd_variants_check_their_workspace(lib):
    atomic = lib.dsa_sparse_attn_bwd_workspace_size_ex(4, 8, 64, 8, 0)
    # enough for the atomic variant, too small for the deterministic one
    rc = lib.dsa_sparse_attn_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, FAKE, NULL, 4, 8, 64, 576, 512, 8, 0.1, FAKE,
                                    FAKE, NULL, 1, FAKE, atomic, NULL)
    assert rc == ops.DSA_ERR_WORKSPACE
    rc = lib.dsa_sparse_attn_bwd_ex(FAKE, FAKE, FAKE, FAKE, FAKE, NULL, FAKE, NULL, 4, 8, 64, 576, 512, 8, 0.1, FAKE,
                                    FAKE, NULL, 0, FAKE, atomic - 1, NULL)
    assert rc == ops.DSA_ERR_WORKSPACE


def test_workspace_size_depends_on_shapes_only(lib):
    a = lib.dsa_indexer_topk_workspace_size(65536, 64, 128, 2048, 65536)
    b = lib.dsa_indexer_topk_workspace_size(65536, 64, 128, 2048, 65536)
    assert a == b and a % 256 == 0


@pytest.mark.parametrize("T,k,s_max", [(65536, 2048, 65536), (4096, 2048, 4096), (256, 64, 256), (1000, 64, 1000),
                                       (16384, 512, 4096), (70001, 256, 70001)])
def test_fused_workspace_layout(lib, T, k, s_max):
    """The fused indexer + top-k workspace: per row four int32 segment counts,
    then per row its final threshold bin (two uint32 keys), then four
    segments of (key, column) pairs, 8 bytes each.  A row holds cap = 4 * min(32 * (ceil(s_max
    / 128) + 1), max(2k, 4096)) pairs: room for every key a tile quarter can
    add to a segment, else a bound at which a segment is cut to its top-k.
    Every part starts on a 256-byte boundary."""
    def a256(x):
        return (x + 255) // 256 * 256

    cap = 4 * min(32 * ((s_max + 127) // 128 + 1), max(2 * k, 4096))
    want = a256(T * 16) + a256(T * 8) + a256(T * cap * 8)
    assert lib.dsa_indexer_topk_workspace_size(T, 64, 128, k, s_max) == want
