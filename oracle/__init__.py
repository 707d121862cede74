"""CPU oracle for the routed-MoE layer.  Test infrastructure only: the
product path never imports this package."""
