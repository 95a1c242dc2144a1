"""GPU parity of the ZeRO-3 gather (and the ZeRO-1/2 full-buffer gather) against the oracle.

The gather is a copy, so the bar is bit-exact on every element.
"""
import numpy as np
import pytest
import torch

import oracle
import sharded_emulated_reduce_gb300 as z

from parity import h16

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def run_gather(n, nd, align, offsets, dst_pad=0, src_pad=0, seed=0):
    """Shards and layer buffers may start `pad` fp16 elements into a larger allocation, to
    exercise relative misalignment of source and destination."""
    np_, s = oracle.partition(n, nd, align)
    g = torch.Generator(device="cuda").manual_seed(seed)
    base = [torch.randint(-32768, 32767, (s + src_pad,), dtype=torch.int16, device="cuda",
                          generator=g) for _ in range(nd)]
    shards = [b[src_pad:] for b in base]
    lens = [offsets[l + 1] - offsets[l] for l in range(len(offsets) - 1)]
    dbase = [torch.full((ln + dst_pad,), -1, dtype=torch.int16, device="cuda") for ln in lens]
    dst = [d[dst_pad:] for d in dbase]
    plan = z.zero_plan_create(n, nd, 3, align, HP)
    z.zero_gather_layers(plan, offsets, shards, [d if d.numel() else None for d in dst])
    assert z.zero_gather_status(plan) == 0
    torch.cuda.synchronize()
    host_shards = [h16(x) for x in shards]
    expected = oracle.gather(host_shards, s, offsets)
    for l, (d, e) in enumerate(zip(dst, expected)):
        assert np.array_equal(h16(d), e), f"layer {l}"
    for d in dbase:  # nothing written before a destination
        assert (h16(d[:dst_pad]) == 0xFFFF).all()
    plan.close()


@pytest.mark.parametrize("n,nd,offsets", [
    (16, 1, [0, 16]),
    (32, 4, [0, 5, 9, 20, 32]),
    (70, 3, [0, 1, 2, 70]),
    (100, 8, [0, 0, 64, 64, 100]),
    (64 * 40, 64, [l * 64 for l in range(41)]),
    (1_000_003, 7, [0, 3, 100_000, 100_007, 555_555, 1_000_003]),
    (10_000_000, 16, [0, 1_234_567, 5_000_000, 9_999_999, 10_000_000]),
])
@pytest.mark.parametrize("dst_pad,src_pad", [(0, 0), (1, 0), (0, 3), (8, 8), (5, 2)])
def test_gather_matches_oracle(n, nd, offsets, dst_pad, src_pad):
    run_gather(n, nd, 8, offsets, dst_pad, src_pad)


@pytest.mark.parametrize("rel", range(1, 8))
def test_relatively_misaligned_source_and_destination(rel):
    # destination buffers start `rel` elements off the source's alignment: every 2-byte
    # relative offset modulo 16 bytes goes through the realigning vector path, over many
    # 64 KiB tiles and their edges
    run_gather(3_000_017, 8, 8, [0, 1_000_001, 1_000_003, 2_345_678, 3_000_017],
               dst_pad=rel, src_pad=0, seed=rel)
    run_gather(700_000, 4, 8, [0, 175_003, 700_000], dst_pad=0, src_pad=rel, seed=10 + rel)


def test_stage2_full_buffer_gather():
    # ZeRO-1/2: one layer [0, N) reassembles the whole fp16 parameter buffer
    run_gather(124_439, 8, 128, [0, 124_439])


def test_many_segments_cross_the_per_launch_table():
    n, nd = 300 * 8 * 64, 64
    offsets = list(range(0, n + 1, n // 300))
    run_gather(n, nd, 8, offsets)


def test_many_segments_of_both_alignment_classes():
    # every other boundary moved by 3 elements: aligned and misaligned segments interleave,
    # and each of the two per-launch tables (bulk-copy kernel, realigning kernel) overflows
    # its 128 entries within one call (about 180 segments each)
    n, nd = 300 * 8 * 64, 64
    step = n // 300
    offsets = [0] + [k * step + (k % 2) * 3 for k in range(1, 300)] + [n]
    run_gather(n, nd, 8, offsets)
    run_gather(n, nd, 8, offsets, dst_pad=3, src_pad=1, seed=7)


def test_prefetch_layers_with_per_layer_events():
    # producer stream gathers layer by layer; a consumer stream waits on each layer's
    # event and reads it (sum of its bits) while later layers are still being gathered
    n, nd = 4_000_000, 16
    np_, s = oracle.partition(n, nd, 8)
    g = torch.Generator(device="cuda").manual_seed(3)
    shards = [torch.randint(-30000, 30000, (s,), dtype=torch.int16, device="cuda", generator=g)
              for _ in range(nd)]
    offs = [l * 400_000 for l in range(11)]
    dst = [torch.empty(offs[l + 1] - offs[l], dtype=torch.int16, device="cuda") for l in range(10)]
    plan = z.zero_plan_create(n, nd, 3, 8, HP)
    producer, consumer = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    events = z.zero_prefetch_layers(plan, offs, shards, dst, producer)
    sums = []
    for l, ev in enumerate(events):
        consumer.wait_event(ev)
        with torch.cuda.stream(consumer):
            sums.append(dst[l].to(torch.int64).sum())
    torch.cuda.synchronize()
    exp = oracle.gather([h16(x) for x in shards], s, offs)
    for l in range(10):
        assert np.array_equal(h16(dst[l]), exp[l])
        assert sums[l].item() == int(exp[l].view(np.int16).astype(np.int64).sum())
    plan.close()


def test_gather_layers_events_misaligned_layers_and_missing_events():
    # odd layer boundaries (both the bulk-copy and the realigning kernel run), a layer
    # without an event, an empty layer; each layer is read on another stream right after
    # its own event, and work enqueued on the call's stream afterwards sees every layer
    n, nd = 3_000_017, 8
    np_, s = oracle.partition(n, nd, 8)
    g = torch.Generator(device="cuda").manual_seed(4)
    shards = [torch.randint(-32768, 32767, (s,), dtype=torch.int16, device="cuda", generator=g)
              for _ in range(nd)]
    offs = [0, 8, 400_003, 400_003, 1_200_000, 1_999_999, 2_400_000, n]
    dst = [torch.full((max(1, offs[l + 1] - offs[l]),), -1, dtype=torch.int16, device="cuda")
           for l in range(len(offs) - 1)]
    plan = z.zero_plan_create(n, nd, 3, 8, HP)
    producer, consumer = torch.cuda.Stream(), torch.cuda.Stream()
    events = z.make_layer_events(len(offs) - 1)
    events[3] = None
    torch.cuda.synchronize()
    z.zero_profile_enable(plan, True)
    z.zero_gather_layers_events(plan, offs, shards, dst, events, producer)
    sums = {}
    for l, ev in enumerate(events):
        if ev is None:
            continue
        consumer.wait_event(ev)
        with torch.cuda.stream(consumer):
            sums[l] = dst[l][:offs[l + 1] - offs[l]].to(torch.int64).sum()
    with torch.cuda.stream(producer):  # after the call on its own stream: all layers
        total = torch.stack([d[:offs[l + 1] - offs[l]].to(torch.int64).sum()
                             for l, d in enumerate(dst)]).sum()
    torch.cuda.synchronize()
    assert z.zero_gather_status(plan) == 0
    launches = z.zero_profile_read(plan)[1][z.PROF_GATHER]
    assert launches >= len(offs) - 2  # one launch (or two) per non-empty layer
    exp = oracle.gather([h16(x) for x in shards], s, offs)
    for l in range(len(offs) - 1):
        got = h16(dst[l])[:offs[l + 1] - offs[l]]
        assert np.array_equal(got, exp[l]), l
        if l in sums:
            assert sums[l].item() == int(exp[l].view(np.int16).astype(np.int64).sum()), l
    assert total.item() == sum(int(e.view(np.int16).astype(np.int64).sum()) for e in exp)
    plan.close()
