// Launch-choice rows per (format class, size bucket), written by tune.py from a timing sweep on
// NVIDIA GB300; regenerate with that script rather than editing by hand.  Rows of one class are in
// ascending key order; a row whose fields are all -1 / 0 keeps the built-in rule.  The sentinel row
// ends the table.
#pragma once
namespace hq {
static const TuneRow kTuneRows[] = {
    {0, 0, 256, {-1, 0, -1, 0, -1, 0}},  // w4a16_asym key (0, 256]: built-in rule
    {0, 0, 512, {0, 256, 0, 0, -1, 0}},  // w4a16_asym key (256, 512]: at most 0.80x the built-in time
    {0, 0, INT64_MAX, {-1, 0, -1, 0, -1, 0}},  // w4a16_asym key (512, INT64_MAX]: built-in rule
    {0, 1, 1, {1, 8, 1, 2, 0, 6}},  // moe_w4a16 key (0, 1]: at most 0.84x the built-in time
    {0, 1, 2, {1, 8, 1, 2, 0, 0}},  // moe_w4a16 key (1, 2]: at most 0.87x the built-in time
    {0, 1, 4, {1, 8, 0, 2, 0, 0}},  // moe_w4a16 key (2, 4]: at most 0.90x the built-in time
    {0, 1, 8, {-1, 0, -1, 0, -1, 0}},  // moe_w4a16 key (4, 8]: built-in rule
    {0, 1, 16, {0, 64, 0, 0, 1, 0}},  // moe_w4a16 key (8, 16]: at most 0.88x the built-in time
    {0, 1, INT64_MAX, {-1, 0, -1, 0, -1, 0}},  // moe_w4a16 key (16, INT64_MAX]: built-in rule
    {1, 0, INT64_MAX, {-1, 0, -1, 0, -1, 0}},  // w8a16 key (0, INT64_MAX]: built-in rule
    {2, 0, 128, {-1, 0, -1, 0, -1, 0}},  // nvfp4 key (0, 128]: built-in rule
    {2, 0, 256, {-1, 64, 0, 0, -1, 0}},  // nvfp4 key (128, 256]: at most 0.93x the built-in time
    {2, 0, 512, {-1, 128, 0, 0, -1, 0}},  // nvfp4 key (256, 512]: at most 0.78x the built-in time
    {2, 0, 1024, {-1, 0, -1, 0, -1, 0}},  // nvfp4 key (512, 1024]: built-in rule
    {2, 0, 2048, {-1, 256, 0, 0, -1, 0}},  // nvfp4 key (1024, 2048]: at most 0.64x the built-in time
    {2, 0, INT64_MAX, {-1, 0, -1, 0, -1, 0}},  // nvfp4 key (2048, INT64_MAX]: built-in rule
    {0, 2, 2, {1, 8, 0, 2, 0, 0}},  // moe_w4a16_down key (0, 2]: at most 0.93x the built-in time
    {0, 2, 8, {-1, 0, -1, 0, -1, 0}},  // moe_w4a16_down key (2, 8]: built-in rule
    {0, 2, 128, {0, 64, 0, 0, 1, 0}},  // moe_w4a16_down key (8, 128]: at most 0.93x the built-in time
    {0, 2, INT64_MAX, {-1, 0, -1, 0, -1, 0}},  // moe_w4a16_down key (128, INT64_MAX]: built-in rule
    {3, 1, 1, {-1, 0, -1, 0, -1, 0}},  // moe_mxfp4 key (0, 1]: built-in rule
    {3, 1, 2, {-1, 64, 0, 0, 1, 0}},  // moe_mxfp4 key (1, 2]: at most 0.97x the built-in time
    {3, 1, 8, {-1, 128, 0, 0, 1, 0}},  // moe_mxfp4 key (2, 8]: at most 0.82x the built-in time
    {3, 1, 32, {-1, 0, -1, 0, -1, 0}},  // moe_mxfp4 key (8, 32]: built-in rule
    {3, 1, 128, {-1, 256, 0, 0, 1, 0}},  // moe_mxfp4 key (32, 128]: at most 0.94x the built-in time
    {3, 1, INT64_MAX, {-1, 0, -1, 0, -1, 0}},  // moe_mxfp4 key (128, INT64_MAX]: built-in rule
    {3, 2, 2, {-1, 0, -1, 0, -1, 0}},  // moe_mxfp4_down key (0, 2]: built-in rule
    {3, 2, 8, {-1, 64, 0, 0, 1, 0}},  // moe_mxfp4_down key (2, 8]: at most 0.85x the built-in time
    {3, 2, INT64_MAX, {-1, 0, -1, 0, -1, 0}},  // moe_mxfp4_down key (8, INT64_MAX]: built-in rule
    {4, 0, INT64_MAX, {-1, 0, -1, 0, -1, 0}},  // w4a8_mx key (0, INT64_MAX]: built-in rule
    {-1, -1, 0, {}},
};
}  // namespace hq
