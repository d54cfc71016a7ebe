"""The algorithmic-byte counts behind the bench's roofline fractions, against
values worked out by hand from the data layout (d = 128, T = 8, bf16 inputs,
fp32 state and outputs, ring depth 8, 32 heads)."""
import bench


def test_spec_verify_unit_bytes():
    # state read 128*128*4; T tokens of q, k, v, alpha (128 bf16 each) + beta;
    # T fp32 outputs of 128; ring write of T entries (k, alpha, v + beta);
    # slot and ctrl words
    base = 65536 + 8 * (4 * 128 * 2 + 2) + 8 * 128 * 4 + 8 * (3 * 128 * 2 + 2) + 8
    assert base == 84008
    assert bench.unit_bytes(0) == base                       # nothing to replay
    assert bench.unit_bytes(3) == base + 65536 + 3 * 770     # write-back + 3 ring reads
    assert bench.unit_bytes(8) == 155704


def test_decode_and_snapshot_unit_bytes():
    assert bench.decode_unit_bytes() == 2 * 65536 + 1026 + 512 + 12
    verify, commit = bench.snapshot_unit_bytes(0)
    assert verify == 65536 + 8208 + 4096 + 8 * 65536 + 4 and commit == 8
    assert bench.snapshot_unit_bytes(5)[1] == 2 * 65536 + 8


def test_state_cache_bytes_per_sequence_layer():
    c = bench.state_cache_bytes()
    assert c["replay_ssm"] == 32 * 65536 + 32 * 8 * 770 + 32 * 8   # 2 294 528
    assert c["direct_snapshots"] == 9 * 32 * 65536                  # 18 874 368
    assert int(46.48 * 2 ** 30 // c["replay_ssm"]) == 21750
    assert int(46.48 * 2 ** 30 // c["direct_snapshots"]) == 2644


def test_serving_schedule_commits_exactly_the_decode_budget():
    import numpy as np
    steps = bench.serving_schedule(np.random.default_rng(0), 5, 40, 0.8802, 8)
    total = np.zeros(5, dtype=np.int64)
    left = set(range(5))
    for live, a in steps:
        assert set(live.tolist()) == left          # every unfinished one, no other
        assert ((a >= 0) & (a <= 8)).all()
        total[live] += a
        left = {int(i) for i in np.nonzero(total < 40)[0]}
    assert (total == 40).all() and not left


def test_serving_verify_bytes_by_hand():
    import numpy as np
    # step 1: both sequences replay nothing; step 2: sequence 0 replays 3,
    # sequence 1 nothing; step 3: sequence 1 alone replays 2
    steps = [(np.array([0, 1]), np.array([3, 0])),
             (np.array([0, 1]), np.array([8, 2])),
             (np.array([1]), np.array([5]))]
    u0, u3, u2 = 84008, 84008 + 65536 + 3 * 770, 84008 + 65536 + 2 * 770
    assert bench.serving_verify_bytes(steps) == (2 * u0 + u3 + u0 + u2) * 32
    assert bench.serving_verify_bytes(steps) == 17758784
