"""Kernel selection on the host: gist_attn_route answers, for each entry point,
which kernel the call would launch, from the same route functions the entry
points dispatch with.  These tests pin the selection rules without a GPU: every
benchmark workload on its intended kernel, the single-pass tensor-core limit
of 288 keys (d = 64), the staged path behind a workspace, the decode kernels'
shape limits and their fallbacks, and the refusals."""
from __future__ import annotations

import pytest

from attention_cached_kv_gb300 import _build, binding, workloads

FWD, WS, FP8, MASS, GMASK = (binding.ENTRY_FWD, binding.ENTRY_FWD_WS, binding.ENTRY_FP8KV,
                             binding.ENTRY_BLOCK_MASS, binding.ENTRY_GIST_MASK)
ENTRIES = (FWD, WS, FP8, MASS, GMASK)
UNSUP = "unsupported"


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return binding.load_library()


def dims(P, l, Hq, Hkv, d, bl, bpp, nb, flags=0):
    return dict(num_pairs=P, n_new=l, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d, block_len=bl,
                blocks_per_pair=bpp, num_blocks=nb, num_layers=1, layer=0, rope_theta=1e4,
                softmax_scale=0.0, flags=flags)


def routes(dm):
    """The route of each entry point, in ENTRIES order ("unsupported" where the
    entry point refuses the shape with GIST_ATTN_ERR_UNSUPPORTED)."""
    out = []
    for e in ENTRIES:
        try:
            out.append(binding.route(dm, e))
        except binding.GistAttnError as err:
            assert err.code == binding.ERR_UNSUPPORTED, (e, err.code)
            out.append(UNSUP)
    return out


# (fwd, fwd_ws, fp8kv, block_mass, gist_mask) per benchmark workload
WORKLOAD_ROUTES = {
    "tiny": ["prefill_tc", "prefill_tc", "prefill_tc", UNSUP, "prefill_stream"],
    "gist": ["prefill_tc", "prefill_tc", "prefill_tc", UNSUP, "prefill_stream"],
    "wide": ["prefill_tc", "prefill_tc", "prefill_tc", UNSUP, "prefill_stream"],
    # 8 + 8 cached keys, 7 heads per KV head: the short decode; no block mass
    # below 33 cached keys with a group
    "qgist": ["decode_short", "decode_short", "decode_short", UNSUP, "prefill_stream"],
    "paged": ["decode_long", "decode_long", "decode_long", "decode_long", "prefill_stream"],
    "paged_gqa": ["decode_gqa", "decode_gqa", "decode_gqa", "decode_gqa", "prefill_stream"],
}


@pytest.mark.parametrize("name", sorted(WORKLOAD_ROUTES))
def test_benchmark_workloads_take_their_kernels(name):
    assert routes(workloads.dims_of(workloads.SPECS[name])) == WORKLOAD_ROUTES[name]


@pytest.mark.parametrize("k,l", [(1, 16), (64, 16), (8, 64), (64, 64), (1, 256), (32, 256)])
def test_sweep_points_up_to_288_keys_run_in_one_tensor_core_pass(k, l):
    dm = workloads.dims_of(workloads.sweep_spec(k, l))
    assert routes(dm)[:3] == ["prefill_tc"] * 3


def test_past_288_keys_the_workspace_entry_stages_and_the_plain_one_streams():
    # k = 64, l = 256: 320 keys
    dm = workloads.dims_of(workloads.sweep_spec(64, 256))
    assert routes(dm) == ["prefill_stream", "staged", UNSUP, UNSUP, "prefill_stream"]
    # one key past the limit, one key within it
    assert routes(dims(4, 256, 14, 2, 64, 33, 1, 4))[:3] == ["prefill_stream", "staged", UNSUP]
    assert routes(dims(4, 256, 14, 2, 64, 32, 1, 4))[:3] == ["prefill_tc"] * 3


def test_d128_past_128_keys_streams():
    # the wide model with l = 256: no staged path at d = 128
    assert routes(dims(4, 256, 32, 8, 128, 8, 1, 4)) == ["prefill_stream", "prefill_stream", UNSUP,
                                                         UNSUP, "prefill_stream"]


def test_offline_pass_routes():
    # 128 items x 1008 tokens, no cache: pre-rotated inputs take the long
    # tensor-core prefill, pre-RoPE ones the staged path behind a workspace
    rot = dims(128, 1008, 14, 2, 64, 0, 0, 0, flags=binding.FLAG_PREROTATED)
    raw = dims(128, 1008, 14, 2, 64, 0, 0, 0)
    assert routes(rot)[:2] == ["prefill_long", "prefill_long"]
    assert routes(raw)[:2] == ["prefill_stream", "staged"]
    assert routes(rot)[4] == routes(raw)[4] == "prefill_stream"


def test_decode_shapes_outside_the_three_decode_kernels():
    # one head per KV head with 40 cached keys: too short for the long decode,
    # too long for the short one, no group for the GQA one
    assert routes(dims(4, 1, 8, 8, 128, 8, 5, 9))[:4] == ["decode", "decode", UNSUP, UNSUP]
    # a group over 4-row blocks: the short decode copies blocks of multiples of 8 rows
    assert routes(dims(4, 1, 4, 2, 64, 4, 4, 9))[:3] == ["decode", "decode", UNSUP]
    # 20 heads per KV head: past every decode kernel, the streaming prefill takes l = 1
    assert routes(dims(4, 1, 40, 2, 64, 16, 4, 9)) == ["prefill_stream", "prefill_stream", UNSUP,
                                                       UNSUP, "prefill_stream"]


def test_decode_kernel_boundaries():
    # 32 cached keys with a group: the short decode; 48: the GQA decode
    assert routes(dims(4, 1, 14, 2, 64, 8, 4, 9))[:3] == ["decode_short"] * 3
    assert routes(dims(4, 1, 14, 2, 64, 16, 3, 9))[:4] == ["decode_gqa"] * 4
    # one head per KV head: the long decode from 64 cached keys
    assert routes(dims(4, 1, 8, 8, 64, 16, 4, 9))[:4] == ["decode_long"] * 4
    # 16 heads per KV head is the largest group either decode kernel takes
    assert routes(dims(2, 1, 32, 2, 128, 16, 5, 9))[:4] == ["decode_gqa"] * 4
    assert routes(dims(2, 1, 34, 2, 128, 16, 5, 9))[3] == UNSUP


def test_refusals_and_empty_calls():
    assert routes(dims(0, 16, 14, 2, 64, 8, 1, 4)) == ["none"] * 5
    assert routes(dims(2, 16, 258, 2, 64, 8, 1, 4)) == [UNSUP] * 5  # 129 heads per KV head
    for e in ENTRIES:
        with pytest.raises(binding.GistAttnError) as err:
            binding.route(dims(4, 0, 14, 2, 64, 8, 1, 4), e)  # no new token
        assert err.value.code == binding.ERR_DIMS
        with pytest.raises(binding.GistAttnError) as err:
            binding.route(dims(4, 16, 14, 2, 96, 8, 1, 4), e)  # head_dim 96
        assert err.value.code == binding.ERR_UNSUPPORTED
    with pytest.raises(binding.GistAttnError) as err:
        binding.route(dims(4, 16, 14, 2, 64, 8, 1, 4), 7)  # not an entry point
    assert err.value.code == binding.ERR_UNSUPPORTED


def test_workspace_is_asked_for_exactly_where_the_staged_path_runs():
    for dm in (workloads.dims_of(workloads.sweep_spec(64, 256)), dims(128, 1008, 14, 2, 64, 0, 0, 0),
               workloads.dims_of(workloads.sweep_spec(32, 256)), dims(4, 256, 32, 8, 128, 8, 1, 4)):
        staged = binding.route(dm, WS) == "staged"
        assert (binding.workspace_bytes(dm) > 0) == staged


def test_gpu_parity_shapes_reach_every_single_launch_kernel():
    """The GPU parity tests' edge shapes, short-cache decodes and GQA decodes,
    routed on the host: between them they run every kernel gist_attn_fwd can
    launch (the long prefill and the staged path have test files of their
    own), so a change of the selection rules cannot leave a kernel untested."""
    import test_parity_gpu as par

    def d(P, l, Hq, Hkv, hd, bl, bpp, nb):
        return dict(dims(P, l, Hq, Hkv, hd, bl, bpp, nb), num_layers=2, layer=1)

    seen = {binding.route(d(*s)) for s in par.EDGE}
    seen |= {binding.route(d(P, 1, Hq, Hkv, hd, bl, bpp, 9)) for P, Hq, Hkv, hd, bl, bpp in par.SHORT}
    seen |= {binding.route(d(P, 1, Hq, Hkv, hd, bl, bpp, 9)) for P, Hq, Hkv, hd, bl, bpp in par.GQA}
    assert seen >= {"prefill_tc", "prefill_stream", "decode_long", "decode_short", "decode_gqa",
                    "decode"}, seen
