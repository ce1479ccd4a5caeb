"""GB300-native dynamic block-sparse attention with a mean-pooled block router."""
