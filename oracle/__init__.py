"""fp64 CPU oracle of the MoE layer: test infrastructure only (tests, smoke check and the
benchmark's CPU baseline). The product path never imports it."""
